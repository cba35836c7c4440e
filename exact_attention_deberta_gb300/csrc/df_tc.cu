// Host orchestration of the tensor-core forward (bf16 / fp16 I/O): the TMA
// tensor maps of every operand and the launch order planning kernel -> near
// tiles -> far tiles on one stream.
//
// Operation: DisentangledFlash README "Status" (C2P/P2C disentangled attention,
// FP16/BF16, factorized padding masks, packed cu_seqlens) and the kernels-community
// "DisentangledFlash" discussion "Motivation" (exact, tiled and streaming, no
// [B,H,L,L] matrix).
//
// The near-tile kernels (df_tc_near64.cu, df_tc_near128.cu) take every tile
// whose relative distances are not all saturated and leave, for query blocks
// that also have far tiles, the un-normalised partial state that the far-tile
// kernel (df_tc_far.cu) continues from; with no far tile possible for the
// batch's lengths the near-tile kernel writes every output row alone.
#include "df_tc_common.cuh"

#include <cudaTypedefs.h>

#include <algorithm>

namespace dfa {

namespace {

using namespace ptx;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Row-major [rows][row_elems] 16-bit matrix in boxes of `inner` x 128 elements:
// 64-element boxes with the 128-byte swizzle, 16-element boxes with the 32-byte one.
bool encode_rows(CUtensorMap* m, const void* base, long long rows, long long row_elems, bool bf16,
                 int inner = 64, int box_rows = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
  const cuuint32_t box[2] = {(cuuint32_t)inner, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_enabled() { return true; }

cudaError_t launch_tc(const Problem& p, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev_mid,
                      cudaEvent_t ev1, int* launches) {
  *launches = 0;
  if (p.T == 0 || p.max_items == 0) return cudaSuccess;
  const bool bf16 = p.dtype == DF_BF16;
  TcMaps maps;
  const long long row = (long long)p.H * p.d;
  if (!encode_rows(&maps.q, p.q, p.T, row, bf16) || !encode_rows(&maps.k, p.k, p.T, row, bf16) ||
      !encode_rows(&maps.v, p.v, p.T, row, bf16) ||
      !encode_rows(&maps.pk, p.pk, 2LL * p.span, row, bf16) ||
      !encode_rows(&maps.pq, p.pq, 2LL * p.span, row, bf16))
    return cudaErrorInvalidValue;
  if (!encode_rows(&maps.kaug, p.kaug, p.T, 16LL * p.H, bf16, 16) ||
      !encode_rows(&maps.kaug_sel, p.kaug_sel, 256, 16, bf16, 16))
    return cudaErrorInvalidValue;
  // the selector rows of the d = 64 near-tile kernel's scalar MMAs: 16 rows per head
  if (p.scal_in_near && (p.d != 64 || !encode_rows(&maps.absel, p.absel, 16LL * p.H, 64, bf16, 64, 16)))
    return cudaErrorInvalidValue;
  if (p.d == 64 || p.d == 128) {
    if (p.n_diag < 1 || !encode_rows(&maps.dpk, p.diag_pk, 128LL * (p.n_diag + 1), row, bf16) ||
        !encode_rows(&maps.dpq, p.diag_pq, 128LL * (p.n_diag + 1), row, bf16))
      return cudaErrorInvalidValue;
  } else {
    maps.dpk = maps.pk;
    maps.dpq = maps.pq;
  }
  if (ev0) cudaEventRecord(ev0, s);
  cudaError_t e;
  e = p.d == 64 ? launch_near64(p, maps, s) : launch_near128(p, maps, s);
  if (ev_mid) cudaEventRecord(ev_mid, s);
  // with no far tile possible the near-tile kernel writes every output row
  if (e == cudaSuccess && p.far_possible) e = launch_far(p, maps, s);
  if (ev1) cudaEventRecord(ev1, s);
  *launches = p.far_possible ? 2 : 1;
  return e;
}

}  // namespace dfa
