// Shared definitions of the disentangled-attention CUDA library (sm_103a).
//
// The operation follows the DisentangledFlash 0.2.0 README ("Status": C2P/P2C
// disentangled attention, factorized 2-D padding masks, packed cu_seqlens
// inference) and the kernels-community "DisentangledFlash" discussion
// ("Motivation": content-to-position and position-to-content terms added to
// the content-to-content score, exact evaluation without the [B,H,L,L] matrix).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "df_attn.h"

namespace dfa {

// Query rows per work item (one tcgen05 M=128 tile).
constexpr int kQBlock = 128;
// Keys per far tile of the tensor-core path.
constexpr int kKBlock = 128;
// Stand-in for -inf in the key-term block (raw score units): it must stay
// finite because the MMA multiplies the unused side's terms by 0.  A masked key
// carries it in both the high and the low part of each side, so the score MMA
// adds 2 x (-65504): the key's weight underflows to 0 as long as the raw scores
// |Q.K + Q.PK + K.PQ| of the row stay well below 131008.
constexpr float kMaskedKeyTerm = -65504.f;

// Workspace views and call parameters handed to every kernel.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const void* pk;
  const void* pq;
  const uint8_t* key_mask;    // padded mode
  const int32_t* cu_seqlens;  // packed mode
  void* out;
  int B, H, L, T, d;
  int buckets, max_rel, span;
  int dtype;                  // df_dtype
  int packed;
  float kscale;               // log2(e) / sqrt(3 d): logits are kept in log2 units
  // workspace sections
  df_ws_header* hdr;
  int32_t* idx;               // [2 lt - 1]
  int4* items;                // [max_items]
  int4* seqs;                 // [B] planner scratch {start, n, nblk, order}
  float* scal;                // [H][4][t_pad]
  float* keybias;             // [t_pad]
  float* partial;             // [T][H][d + 2]
  int max_items;
  int t_pad;
  int lt;                     // index-table half width: idx of r at r + lt - 1, |r| < lt
  // diagonal position tables (d = 64, 128): row (m - diag_m0) * 256 + t holds
  // PK / PQ[idx(128 m - 127 + t)], [rows][H][d] in the I/O type
  void* diag_pk;
  void* diag_pq;
  // far tiles: per (key, head) 16 values (beta_neg hi, lo, beta_pos hi, lo, 0...)
  // in the I/O type, and the two selector blocks [256][16]
  void* kaug;
  void* kaug_sel;
  // [H][16][64] in the I/O type: PK[0], PK[top], PQ[0], PQ[top] of each head
  // (then zeros), the B operand of the d = 64 near-tile kernel's scalar MMAs
  void* absel;
  int n_diag;
  int diag_m0;
  unsigned long long wait_budget;
  int zero_out;               // the planner zeroes the output rows of masked tokens
  int far_possible;           // 0: no tile of any sequence (length <= L) is a far tile
  int scal_needed;            // 0: no 64 x 64 tile is far either, so no kernel reads the
                              //    per-token scalars or the key-term block
  int scal_in_near;           // 1: the d = 64 near-tile kernel writes the far tiles'
                              //    query scalars and key-term blocks (the planner
                              //    only writes the selector-row table)
};

// Views of the backward pass (gradients in fp32).
struct BwdProblem {
  Problem f;                  // the forward's inputs and planning views
  const void* dout;           // [tokens][H][d], the I/O type
  float* dq;                  // [tokens][H][d]
  float* dk;
  float* dv;
  float* dpk;                 // [2 span][H][d]
  float* dpq;
  float* lse;                 // [T][H] row log-sum-exp of the logits (log2 units); +inf: no output
  float* drow;                // [T][H] dO_i . O_i
  float* gc;                  // [T][H][R] sums of dS along each query row, by relative index
  float* gp;                  // [T][H][R] the same along each key column
  float* part;                // [2][splits][H][R][d] partial position gradients
  int R;                      // 2 span
  int splits;                 // token ranges of the position-gradient reduction
  int kchunk;                 // tokens per range
  float sscale;               // 1 / sqrt(3 d)
};

// DeBERTa log-bucketed relative position.  The identity inside |r| <= mid;
// logarithmic growth that reaches 2 mid - 1 at |r| = max_rel - 1 outside it.
// Evaluated in double precision (CUDA's log) so that no bucket edge moves.
__device__ __forceinline__ int rel_bucket(int r, int buckets, int max_rel) {
  if (buckets <= 0) return r;
  const int mid = buckets / 2;
  const int a = r < 0 ? -r : r;
  if (a <= mid) return r;
  const double f = log((double)a / (double)mid) / log((double)(max_rel - 1) / (double)mid);
  const int g = (int)ceil(f * (double)(mid - 1)) + mid;
  return r < 0 ? -g : g;
}

__device__ __forceinline__ int rel_index(int r, int buckets, int max_rel, int span) {
  int u = rel_bucket(r, buckets, max_rel) + span;
  u = u < 0 ? 0 : u;
  return u > 2 * span - 1 ? 2 * span - 1 : u;
}

template <typename T> struct IO;
template <> struct IO<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct IO<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <> struct IO<__half> {
  static __device__ __forceinline__ float load(const __half* p) { return __half2float(*p); }
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

// Staging of [rows][ts] token-major tiles into shared memory as fp32 with
// 16-byte global loads (each row's columns start 16-byte aligned).
// Transposed: dst[c * STRIDE + r] for columns c < C; with STRIDE = 1 modulo 32
// the scalar stores of a warp fall in 32 different banks.
template <typename T, int C, int STRIDE, int NT>
__device__ __forceinline__ void stage_transposed(const T* __restrict__ base, size_t ts, int rows, int lim,
                                                 float* dst) {
  constexpr int V = 16 / sizeof(T), VPR = C / V;
  static_assert(C % V == 0 && STRIDE % 32 == 1, "16-byte rows, conflict-free stores");
  for (int e = threadIdx.x; e < rows * VPR; e += NT) {
    const int r = e / VPR, v = e % VPR;
    float f[V];
    if (r < lim) {
      const uint4 raw = *reinterpret_cast<const uint4*>(base + (size_t)r * ts + v * V);
      const T* el = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int k = 0; k < V; ++k) f[k] = IO<T>::to_f(el[k]);
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k) f[k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < V; ++k) dst[(v * V + k) * STRIDE + r] = f[k];
  }
}

// Row-major: dst[r * C + c] (dst 16-byte aligned), 16-byte loads and stores.
template <typename T, int C, int NT>
__device__ __forceinline__ void stage_rows(const T* __restrict__ base, size_t ts, int rows, int lim,
                                           float* dst) {
  constexpr int V = 16 / sizeof(T), VPR = C / V;
  static_assert(C % V == 0 && V % 4 == 0, "16-byte rows");
  for (int e = threadIdx.x; e < rows * VPR; e += NT) {
    const int r = e / VPR, v = e % VPR;
    float4 f[V / 4];
    if (r < lim) {
      const uint4 raw = *reinterpret_cast<const uint4*>(base + (size_t)r * ts + v * V);
      const T* el = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int k = 0; k < V / 4; ++k)
        f[k] = make_float4(IO<T>::to_f(el[4 * k]), IO<T>::to_f(el[4 * k + 1]), IO<T>::to_f(el[4 * k + 2]),
                           IO<T>::to_f(el[4 * k + 3]));
    } else {
#pragma unroll
      for (int k = 0; k < V / 4; ++k) f[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < V / 4; ++k) reinterpret_cast<float4*>(dst + (size_t)r * C + v * V)[k] = f[k];
  }
}

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void raise_device_error(df_ws_header* hdr, int code, int where) {
  if (atomicCAS(&hdr->status, 0, code) == 0) hdr->status_where = where;
}

// Programmatic dependent launch.  The planning kernel lets the attention
// kernel after it be scheduled early; that kernel sets up its shared memory,
// barriers and tensor memory, then waits here for the planning grid to finish
// (and its writes to be visible) before its first global-memory access.  The
// wait returns at once for a launch without the programmatic attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` on `s` with the programmatic-serialisation attribute: it
// may start while the kernel before it on the stream is still running, and
// must call grid_dependency_wait() before it touches global memory.
template <typename... Params, typename... Args>
cudaError_t launch_after_plan(void (*kernel)(Params...), int grid, int threads, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace dfa

// Host-side launchers (defined in the .cu files).
namespace dfa {
cudaError_t launch_plan(const Problem& p, cudaStream_t s);
cudaError_t launch_index_table(int buckets, int max_rel, int span, int max_len, int32_t* idx,
                               cudaStream_t s);
cudaError_t launch_simt(const Problem& p, cudaStream_t s, int* launches);
cudaError_t launch_pad32(const void* const src[5], void* const dst[5], const long long rows[5],
                         cudaStream_t s);
cudaError_t launch_unpad32(const void* src, void* dst, long long rows, cudaStream_t s);
// Fast fp32 mode: fp32 -> fp16 copies of five arrays (n values each, a multiple
// of 4; *flag set to 1 if a value is out of fp16's range), and fp16 -> fp32 of
// the output (DF_ERR_INVALID_ARG recorded in the status word at hdr if *flag).
cudaError_t launch_to_half(const float* const src[5], void* const dst[5], const long long n[5], int* flag,
                           cudaStream_t s);
cudaError_t launch_to_float(const void* src, float* dst, long long n, const int* flag, void* hdr,
                            cudaStream_t s);
cudaError_t launch_bwd(const BwdProblem& b, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev_mid,
                       cudaEvent_t ev1, int* launches);
}  // namespace dfa
