// Pieces shared by the two tensor-core kernels (near tiles, far tiles).
#pragma once

#include <cuda.h>

#include "df_common.cuh"
#include "df_tc_ptx.cuh"

namespace dfa {

constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column box of 16-bit values
constexpr unsigned long long kDrainBudget = 1ull << 31;

struct TcMaps {
  CUtensorMap q, k, v, pk, pq;
  CUtensorMap dpk, dpq;        // diagonal position tables (near tiles)
  CUtensorMap kaug, kaug_sel;  // far tiles: key-term block and selector rows (16 wide)
  CUtensorMap absel;           // d = 64 near tiles: PK / PQ rows of the far-tile terms (16 x 64 boxes)
};

constexpr uint32_t kAugBytes = 128 * 16 * 2;  // one 128-row x 16-column 16-bit box

// Tensor-memory column maps are checked at compile time: every region (first
// column, width in 32-bit columns) must end inside the kernel's allocation.
constexpr bool tmem_region_fits(uint32_t first, uint32_t width, uint32_t alloc) {
  return width > 0 && first + width <= alloc;
}

// Descriptor of a K-major 128-row operand with 16 elements (32 bytes) per row,
// 32-byte swizzle: 8-row groups 256 bytes apart.
__device__ __forceinline__ uint64_t aug_desc(const uint8_t* tile) {
  uint64_t d = (uint64_t)((ptx::smem_u32(tile) >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;           // leading byte offset (unused by a single K step)
  d |= (uint64_t)(256 >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1 << 46;           // descriptor version of tcgen05
  d |= (uint64_t)6 << 61;           // 32-byte swizzle
  return d;
}

// K step ks (16 elements) of a K-major 128-row tile stored as 64-column,
// 128-byte-swizzled boxes: box ks/4, 32-byte offset inside it.
__device__ __forceinline__ uint64_t kmajor_desc(const uint8_t* tile, int ks) {
  return ptx::sdesc_sw128(ptx::smem_u32(tile + (ks >> 2) * kBoxBytes + (ks & 3) * 32), 16, 1024);
}

// Offset of K step ks from step 0 in a descriptor's 16-byte address field, so
// that the descriptors of one tile are a base plus compile-time constants.
__host__ __device__ constexpr uint64_t kmajor_step(int ks) {
  return (uint64_t)(((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t vtile_step(int ks) { return (uint64_t)(ks * 2048 >> 4); }

// K step ks (16 key rows) of a 128-row V tile used as the MN-major B operand of
// P.V: 16 rows x 128 B = 2048 B per step, 64-column boxes kBoxBytes apart.
__device__ __forceinline__ uint64_t vtile_desc(uint32_t v_addr, int ks) {
  return ptx::sdesc_sw128(v_addr + ks * 2048, kBoxBytes, 1024);
}

// Key blocks of query block i0 whose 128 x 128 tile is near (its relative
// distances i - j in [i0 - j0 - 127, i0 - j0 + 127] are not all saturated).
// The near blocks form one run [*jlo, *jhi); blocks before it are saturated on
// the positive side (idx = 2 span - 1), blocks after it on the negative side.
// Block jb is saturated on the positive side iff i0 - 128 jb - 127 >= rsp, i.e.
// jb <= floor((i0 - 127 - rsp) / 128); it is short of saturation on the
// negative side iff i0 - 128 jb + 127 > rsn, i.e. jb < ceil((i0 + 127 - rsn) / 128).
// (Arithmetic right shifts give the floor of a negative numerator.)
__device__ __forceinline__ void near_block_range(int i0, int nkb, int rsp, int rsn, int* jlo,
                                                 int* jhi) {
  int lo = ((i0 - 127 - rsp) >> 7) + 1;
  int hi = -((rsn - i0 - 127) >> 7);
  lo = lo < 0 ? 0 : (lo > nkb ? nkb : lo);
  hi = hi < 0 ? 0 : (hi > nkb ? nkb : hi);
  *jlo = lo;
  *jhi = hi > lo ? hi : lo;
}

// Partial softmax state handed from the near-tile kernel to the far-tile kernel:
// un-normalised O rows (fp32) and (running max, running sum) per (token, head).
__device__ __forceinline__ float* partial_o(const Problem& p) { return p.partial; }
__device__ __forceinline__ float2* partial_ml(const Problem& p) {
  return reinterpret_cast<float2*>(p.partial + (size_t)p.B * p.L * p.H * p.d);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

cudaError_t launch_far(const Problem& p, const TcMaps& maps, cudaStream_t s);
cudaError_t launch_near64(const Problem& p, const TcMaps& maps, cudaStream_t s);
cudaError_t launch_near128(const Problem& p, const TcMaps& maps, cudaStream_t s);

// Bounded wait that also gives up as soon as another role of the CTA has
// aborted.  On a timeout it records DF_ERR_DEVICE_TIMEOUT and raises the CTA's
// abort flag.  Callers keep their control flow identical after a failure (no
// early exit), so that warp-collective instructions and named barriers stay
// matched.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              unsigned long long budget, volatile int* abort,
                                              df_ws_header* hdr, int where) {
  // a completed phase is a valid result even while the CTA aborts
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (*abort) return false;
    if ((unsigned long long)(clock64() - t0) > budget) {
      *abort = 1;
      raise_device_error(hdr, DF_ERR_DEVICE_TIMEOUT, where);
      return false;
    }
    if (ptx::mbar_try_wait(bar, parity)) return true;
  }
}

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace dfa
