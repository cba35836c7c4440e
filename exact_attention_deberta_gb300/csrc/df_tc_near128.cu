// Near-tile fused forward for head size 128 on tcgen05 (bf16 / fp16 I/O; fp32
// accumulation and fp32 position terms).
//
// Operation: DisentangledFlash README "Status" (C2P/P2C disentangled attention,
// FP16/BF16, packed cu_seqlens, head dimensions 32, 64 and 128) and the
// kernels-community "DisentangledFlash" discussion "Motivation" (exact, tiled
// and streaming, no [B,H,L,L] matrix).
//
// The position terms take the diagonal form of the head-size-64 kernel.  In a
// 128 x 128 tile with query block i0 and key block j0 = i0 - 128 m, element
// (i', j') has relative distance r = 128 m - 127 + t, t = i' - j' + 127 its
// diagonal.  The planning kernel's diagonal tables hold, per offset m, the PK
// and PQ rows at idx(r) for every diagonal, so that MMAs give
//     C[i'][t] = Q_i . PK[idx(r_t)]      P[j'][t] = K_j . PQ[idx(r_t)]
// in two halves of 128 diagonals each (C0, C1, P0, P1: 128 x 128 x 128 MMAs),
// and the score element needs C[i'][i' - j' + 127] + P[j'][i' - j' + 127].
//
// At head size 128 the operands take twice the shared memory (a 128-row tile
// is 32 KB), so there is room for ONE fp32 skew buffer W [128][132] instead of
// one per term.  Every tile sums the two terms in it:
//   1. the C products are drained by query row: lane i' stores diagonal t at
//      W[i'][i' + 127 - t] (its own row; quarter q fills rows 32 q .. +31);
//   2. after a barrier of the compute warps, the P products are drained by key
//      row: lane j' adds diagonal t (plus the key's bias) to W[t - 127 + j'][j']
//      (quarter q updates key columns 32 q .. +31 of every row; each element
//      has one writer, so a plain load, add and store);
//   3. each warp reads its 32 keys of its rows, C + P, once quarter g (the
//      owner of its key columns) has added its P terms.
// Rows of 132 words keep the drains and the row reads free of bank conflicts
// (word 133 i' + const for the 32 lanes of a store; rows an odd number of
// 16-byte units apart for the row reads).  Holding the C terms in W rather
// than in registers keeps the compute warps within 96 registers.
//
// Tensor memory: two 128-column slots take the products in the order C0, C1,
// P0, P1, S of every tile (product x in slot x mod 2), so that the tensor core
// computes the next product while the current one is drained; O 256-383; Q
// (16-bit pairs, the A operand of C0, C1 and S) 384-447; P (16-bit pairs, the
// A operand of P.V) 448-511.  P has its own columns so that the next tile's
// products do not wait for P.V.
//
// Roles (one CTA per SM, persistent over the work list):
//   warps 0-15  compute: warp w owns TMEM lanes 32 (w % 4) .. +31 (query rows
//               for C, S and O; key rows for P) and score columns
//               32 (w / 4) .. +31 of every tile; they drain the position
//               products, gather, run the online softmax and write P;
//   warp 16     MMA issue (one thread);
//   warp 17     TMA loads (one thread): the diagonal-table halves through a
//               two-buffer ring, K, V; it also claims the work items (longest
//               first, one global counter) and hands them to the other roles.
// A masked or absent key is masked through its P row: the P drains add the
// key's bias (0 or -inf) to every position term they store for it.
//
// A query block whose key range also has far tiles leaves its un-normalised
// partial state (O, running max, running sum) for the far-tile kernel;
// otherwise this kernel writes the final rows.
#include "df_tc_common.cuh"

#include <algorithm>
#include <type_traits>

namespace dfa {

namespace {

using namespace ptx;

constexpr int kD = 128;
constexpr int kTile = 128;
constexpr int kChunks = kD / 64;                // 64-column boxes per 128-row operand tile
constexpr uint32_t kTileBytes = kChunks * kBoxBytes;  // 32 KB
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 64;  // + the MMA warp and the load warp
constexpr uint32_t kRowW = 132;                 // words per W row: 128 keys + 4 of padding
constexpr uint32_t kRowB = kRowW * 4;           // 528 bytes
static_assert((kRowW + 1) % 2 == 1 && (kRowB / 16) % 2 == 1, "conflict-free drains and gathers");
static_assert(kD * 4 <= kRowB, "an fp32 O row fits a W row");

// Tensor-memory columns.
constexpr uint32_t kSlots = 2, kSlotCols = 128;
constexpr uint32_t kColO = kSlots * kSlotCols;  // 256
constexpr uint32_t kColQ = kColO + kD;          // 384
constexpr uint32_t kColP = kColQ + kD / 2;      // 448
static_assert(tmem_region_fits(0, kSlots * kSlotCols, kColO), "product slots below O");
static_assert(tmem_region_fits(kColO, kD, kColQ), "O below Q");
static_assert(tmem_region_fits(kColQ, kD / 2, kColP), "Q below P");
static_assert(tmem_region_fits(kColP, kTile / 2, 512), "P inside 512 columns");
constexpr uint32_t kRing = 2;      // diagonal-table halves in flight
constexpr uint32_t kItemRing = 4;  // work items handed from the load warp to the others

struct Smem {
  static constexpr uint32_t k = 0;                        // K tile
  static constexpr uint32_t v = k + kTileBytes;           // V tile
  static constexpr uint32_t e = v + kTileBytes;           // [kRing] diagonal-table halves
  static constexpr uint32_t w = e + kRing * kTileBytes;   // fp32 [128][132] skew buffer
  static constexpr uint32_t red = w + 128 * kRowB;        // float [3][4][128]: row max / sum exchange
  static constexpr uint32_t bars = red + 3 * 4 * 128 * 4;
  static constexpr int kBars = 19 + 2 * kItemRing;
  static constexpr uint32_t misc = bars + kBars * 8;      // abort flag, TMEM slot
  static constexpr uint32_t next = (misc + 16 + 15) & ~15u;  // int4: the compute warps' next item
  static constexpr uint32_t ring = next + 16;                // int4 [kItemRing]: items handed out
  static constexpr uint32_t bytes = ring + 16 * kItemRing;
};
static_assert(Smem::next % 16 == 0 && Smem::ring % 16 == 0 && Smem::w % 16 == 0,
              "16-byte aligned vector regions");
static_assert(Smem::bytes <= 227 * 1024, "near-tile shared memory");
static_assert(Smem::bars % 8 == 0 && Smem::e % 1024 == 0 && Smem::v % 1024 == 0, "alignment");

// Run of 8-column groups (first group, count) that warp g of lane quarter qd
// drains from a position product: term 0 is C (query rows), term 1 is P (key
// rows); half 0 holds diagonals 0..127, half 1 diagonals 128..255.  Lane
// quarter qd needs diagonals [32 qd, 32 qd + 159] of C and [96 - 32 qd,
// 255 - 32 qd] of P; each product's groups are split into four equal runs
// (10 groups per warp per tile).
__device__ __forceinline__ void drain_run(int term, int half, int qd, int g, int* first, int* count) {
  int lo, len;
  if (term == 0) {
    if (half == 0) { lo = 4 * qd; len = 4 - qd; }   // t in [32 qd, 128)
    else { lo = 0; len = qd + 1; }                  // t in [128, 160 + 32 qd)
  } else {
    if (half == 0) { lo = 12 - 4 * qd; len = 1 + qd; }  // t in [96 - 32 qd, 128)
    else { lo = 0; len = 4 - qd; }                      // t in [128, 256 - 32 qd)
  }
  *first = lo + g * len;
  *count = len;
}

// Skew stores of one 8-diagonal run, each made only when its key (row) lies in
// 0 .. 127.  C: value e to key j0 - e of the lane's row, i.e. byte offset
// 4 (7 - e) from the run's lowest key (a7); P: value e to row i0 + e of the
// lane's key column (offset kRowB e from a0).  The base addresses stay inside
// the shared window even where a run starts outside the tile.
__device__ __forceinline__ void st_run_c(uint32_t a7, const uint32_t* r, int j0) {
#define DFA_C(e) sts32_below_at<4 * (7 - e)>(a7, r[e], (uint32_t)(j0 - (e)), 128u);
  DFA_C(0) DFA_C(1) DFA_C(2) DFA_C(3) DFA_C(4) DFA_C(5) DFA_C(6) DFA_C(7)
#undef DFA_C
}
// P: value e (plus the key bias) is added to W at row i0 + e of the lane's key
// column (offset kRowB e from a0), where the C drain stored that element's C
// term; only rows in 0 .. 127.  Each element has exactly one writer, so the
// read-modify-write needs no atomics; one block of PTX, so that the eight loads
// are issued before the first add.
__device__ __forceinline__ void add_run_p(uint32_t a0, const uint32_t* r, float kbias, int i0) {
  static_assert(kRowB == 528, "row stride in the PTX below");
  asm volatile(
      "{\n\t.reg .pred q<8>;\n\t.reg .f32 w<8>, v<8>;\n\t"
      "setp.lt.u32 q0, %0, 128;\n\t"
      "setp.lt.u32 q1, %1, 128;\n\t"
      "setp.lt.u32 q2, %2, 128;\n\t"
      "setp.lt.u32 q3, %3, 128;\n\t"
      "setp.lt.u32 q4, %4, 128;\n\t"
      "setp.lt.u32 q5, %5, 128;\n\t"
      "setp.lt.u32 q6, %6, 128;\n\t"
      "setp.lt.u32 q7, %7, 128;\n\t"
      "@q0 ld.shared.f32 w0, [%8+0];\n\t"
      "@q1 ld.shared.f32 w1, [%8+528];\n\t"
      "@q2 ld.shared.f32 w2, [%8+1056];\n\t"
      "@q3 ld.shared.f32 w3, [%8+1584];\n\t"
      "@q4 ld.shared.f32 w4, [%8+2112];\n\t"
      "@q5 ld.shared.f32 w5, [%8+2640];\n\t"
      "@q6 ld.shared.f32 w6, [%8+3168];\n\t"
      "@q7 ld.shared.f32 w7, [%8+3696];\n\t"
      "add.f32 v0, %10, %9;\n\tadd.f32 w0, w0, v0;\n\t"
      "add.f32 v1, %11, %9;\n\tadd.f32 w1, w1, v1;\n\t"
      "add.f32 v2, %12, %9;\n\tadd.f32 w2, w2, v2;\n\t"
      "add.f32 v3, %13, %9;\n\tadd.f32 w3, w3, v3;\n\t"
      "add.f32 v4, %14, %9;\n\tadd.f32 w4, w4, v4;\n\t"
      "add.f32 v5, %15, %9;\n\tadd.f32 w5, w5, v5;\n\t"
      "add.f32 v6, %16, %9;\n\tadd.f32 w6, w6, v6;\n\t"
      "add.f32 v7, %17, %9;\n\tadd.f32 w7, w7, v7;\n\t"
      "@q0 st.shared.f32 [%8+0], w0;\n\t"
      "@q1 st.shared.f32 [%8+528], w1;\n\t"
      "@q2 st.shared.f32 [%8+1056], w2;\n\t"
      "@q3 st.shared.f32 [%8+1584], w3;\n\t"
      "@q4 st.shared.f32 [%8+2112], w4;\n\t"
      "@q5 st.shared.f32 [%8+2640], w5;\n\t"
      "@q6 st.shared.f32 [%8+3168], w6;\n\t"
      "@q7 st.shared.f32 [%8+3696], w7;\n\t"
      "}\n" ::"r"((uint32_t)i0), "r"((uint32_t)(i0 + 1)), "r"((uint32_t)(i0 + 2)),
      "r"((uint32_t)(i0 + 3)), "r"((uint32_t)(i0 + 4)), "r"((uint32_t)(i0 + 5)),
      "r"((uint32_t)(i0 + 6)), "r"((uint32_t)(i0 + 7)), "r"(a0), "f"(kbias),
      "f"(__uint_as_float(r[0])), "f"(__uint_as_float(r[1])), "f"(__uint_as_float(r[2])),
      "f"(__uint_as_float(r[3])), "f"(__uint_as_float(r[4])), "f"(__uint_as_float(r[5])),
      "f"(__uint_as_float(r[6])), "f"(__uint_as_float(r[7]))
      : "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_near128_kernel(const Problem p, const __grid_constant__ TcMaps maps) {
  using SL = Smem;
  constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, kD, BF16 ? 1 : 0, 0, 1);
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    grid_dependency_wait();
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(p.hdr, DF_ERR_CUDA, 400);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm + SL::k;
  uint8_t* sV = sm + SL::v;
  uint8_t* sE = sm + SL::e;
  float* sRed = reinterpret_cast<float*>(sm + SL::red);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SL::bars);
  uint64_t* q_full = bars + 0;      // Q of the item in TMEM (one arrival per compute warp)
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 2;     // S of the tile done (its last reader of K)
  uint64_t* v_full = bars + 3;
  uint64_t* e_full = bars + 4;      // [kRing]
  uint64_t* e_empty = bars + 6;     // [kRing] the product that read the half is done
  uint64_t* slot_full = bars + 8;   // [2] product in the slot computed
  uint64_t* slot_empty = bars + 10; // [2] product drained (one arrival per compute warp)
  uint64_t* p_full = bars + 12;     // P of the tile in TMEM (one arrival per compute warp)
  uint64_t* pv_done = bars + 13;    // P.V of the tile done (O and P free, V free)
  uint64_t* bar_end = bars + 14;    // every MMA done (exit)
  // Quarter q's P terms are added to W (key columns 32 q .. +31 of every row):
  // one phase per tile, every thread of the quarter's four warps arrives.
  uint64_t* p_drained = bars + 15;  // [4]
  // Work items: the load warp takes the next item of the list (a global
  // counter, longest items first) and hands it to the MMA warp and the compute
  // warps through a ring of kItemRing slots; a slot is free again once both
  // have read it.  An item with n < 0 ends the CTA's list.
  uint64_t* item_full = bars + 19;  // [kItemRing]
  uint64_t* item_empty = bars + 19 + kItemRing;  // [kItemRing] (MMA thread and compute thread 0)
  int4* s_ring = reinterpret_cast<int4*>(sm + SL::ring);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SL::misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < SL::kBars; ++b) mbar_init(bars + b, 1);
    for (uint32_t s = 0; s < kSlots; ++s) mbar_init(slot_empty + s, kComputeWarps);
    mbar_init(p_full, kComputeWarps);
    mbar_init(q_full, kComputeWarps);
    for (uint32_t s = 0; s < kItemRing; ++s) mbar_init(item_empty + s, 2);
    for (int q = 0; q < 4; ++q) mbar_init(p_drained + q, 128);
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == kComputeWarps) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  grid_dependency_wait();  // the planner's outputs (first global access below)
  const uint32_t tO = tmem + kColO, tQ = tmem + kColQ, tP = tmem + kColP;

  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const unsigned long long budget = p.wait_budget;
  df_ws_header* hdr = p.hdr;

  auto wt = [&](uint64_t* bar, uint32_t parity, int where) {
    return wait_or_abort(bar, parity, budget, s_abort, hdr, where);
  };
  if (warp == kComputeWarps) {
    // ================================================================ MMA issue
    if (lane == 0) {
      // Products and P.V issued, tables consumed.  The n-th commit on a barrier
      // completes its phase n, parity n & 1.
      uint32_t ec_n = 0, pp = 0, pv_n = 0, k_n = 0, v_n = 0, q_n = 0;
      bool have_prev = false, prev_first = false;
      const uint64_t dk = kmajor_desc(sK, 0);
      const uint32_t dv_addr = smem_u32(sV);

      // Position product of term `term` (0: C = Q.table with Q from tensor
      // memory, 1: P = K.table) into the next slot, from the next table half.
      auto issue_pos = [&](int term, int where) {
        const uint32_t x = pp, s = x % kSlots, b = ec_n % kRing;
        bool ok = !*s_abort;
        if (ok && x >= kSlots) ok = wt(slot_empty + s, ((x / kSlots) - 1) & 1, where);
        ok = wt(e_full + b, (ec_n / kRing) & 1, where + 1) && ok;
        if (!ok) return;
        tc_fence_after();
        const uint64_t db = kmajor_desc(sE + b * kTileBytes, 0);
        const uint32_t d = tmem + s * kSlotCols;
        if (term) {
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_ss(d, dk + kmajor_step(k), db + kmajor_step(k), kIdescQK, k > 0);
        } else {
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_ts(d, tQ + 8 * k, db + kmajor_step(k), kIdescQK, k > 0 ? 1u : 0u);
        }
        mma_commit(slot_full + s);
        mma_commit(e_empty + b);
        ++pp;
        ++ec_n;
      };
      // O (+)= P.V of the previous tile (P: keys 16 k .. 16 k + 15 at columns
      // 8 k .. 8 k + 7 of the P region).
      auto issue_pv = [&](bool first, int where) {
        bool ok = wt(p_full, pv_n & 1, where);
        ok = wt(v_full, v_n & 1, where + 1) && ok;
        if (!ok) return;
        ++v_n;
        tc_fence_after();
        const uint64_t dv = vtile_desc(dv_addr, 0);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_ts(tO, tP + 8 * k, dv + vtile_step(k), kIdescPV, (!first || k > 0) ? 1u : 0u);
        mma_commit(pv_done);
        ++pv_n;
      };

      for (uint32_t ic = 0;; ++ic) {
        const uint32_t slot = ic % kItemRing;
        if (!wt(item_full + slot, (ic / kItemRing) & 1, 441)) break;
        const int4 item = s_ring[slot];
        mbar_arrive(item_empty + slot);
        if (item.y < 0) break;
        const int n = item.y, ib = item.w;
        const int nkb = (n + kTile - 1) / kTile;
        int jlo, jhi;
        near_block_range(ib * kTile, nkb, rsp, rsn, &jlo, &jhi);
        const int nt = jhi - jlo;
        if (nt <= 0) continue;
        for (int t = 0; t < nt; ++t) {
          // The previous tile's P.V goes first at an item's first tile: the
          // compute warps store this item's Q once that P.V is done.
          if (t == 0) {
            if (have_prev) issue_pv(prev_first, 420);
            wt(q_full, q_n & 1, 404);
            ++q_n;
          }
          issue_pos(0, 410);  // C0
          issue_pos(0, 412);  // C1
          if (t > 0) issue_pv(prev_first, 420);
          wt(k_full, k_n & 1, 405);
          ++k_n;
          issue_pos(1, 414);  // P0
          issue_pos(1, 416);  // P1
          // S = Q.K^T into the next slot
          {
            const uint32_t x = pp, s = x % kSlots;
            bool ok = !*s_abort;
            if (ok && x >= kSlots) ok = wt(slot_empty + s, ((x / kSlots) - 1) & 1, 418);
            if (ok) {
              tc_fence_after();
              const uint32_t d = tmem + s * kSlotCols;
#pragma unroll
              for (int k = 0; k < kD / 16; ++k)
                mma_ts(d, tQ + 8 * k, dk + kmajor_step(k), kIdescQK, k > 0 ? 1u : 0u);
              mma_commit(slot_full + s);
              mma_commit(k_empty);
              ++pp;
            }
          }
          have_prev = true;
          prev_first = t == 0;
        }
      }
      if (have_prev) issue_pv(prev_first, 422);
      // no MMA may still be in flight when the CTA leaves
      mma_commit(bar_end);
      mbar_wait(bar_end, 0, kDrainBudget);
    }
  } else if (warp == kComputeWarps + 1) {
    // ================================================================ loads
    // One thread issues every TMA load, in the order in which the MMAs free
    // the buffers (C0, C1, P0, P1 tables of a tile through the two-buffer ring;
    // K once the previous S is done; V one tile late, once the P.V before it is
    // done), so that no load waits behind another's condition.
    if (lane == 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dpk);
      tma_prefetch_desc(&maps.dpq);
      uint32_t k_n = 0, v_n = 0, e_n = 0;
      int v_head = 0, v_row = 0;
      bool v_pending = false;
      // a 128-row x 128-column tile: two 64-column boxes on one barrier
      auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, int col, int row, uint64_t* bar) {
        mbar_expect_tx(bar, kTileBytes);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kBoxBytes, map, col + 64 * c, row, bar);
      };
      auto e_load = [&](const CUtensorMap* map, int head, int row, int where) {
        const uint32_t b = e_n % kRing;
        bool ok = !*s_abort;
        if (ok && e_n >= kRing) ok = wt(e_empty + b, ((e_n / kRing) - 1) & 1, where);
        if (ok) {
          load_tile(sE + b * kTileBytes, map, head * kD, row, e_full + b);
          ++e_n;
        }
      };
      // V of the previous tile, once the P.V before it is done
      auto v_load = [&](int where) {
        bool ok = !*s_abort;
        if (ok && v_n > 0) ok = wt(pv_done, (v_n - 1) & 1, where);
        if (ok) {
          load_tile(sV, &maps.v, v_head * kD, v_row, v_full);
          ++v_n;
        }
        v_pending = false;
      };
      for (uint32_t ic = 0;; ++ic) {
        // the next item of the list, claimed once its ring slot is free and
        // handed to the other roles
        const uint32_t slot = ic % kItemRing;
        if (ic >= kItemRing && !wt(item_empty + slot, ((ic / kItemRing) - 1) & 1, 440)) break;
        if (*s_abort) break;
        const int it = atomicAdd(&hdr->next_item, 1);
        const int4 item = it < n_items ? p.items[it] : make_int4(-1, -1, -1, -1);
        s_ring[slot] = item;
        mbar_arrive(item_full + slot);  // release: the slot's contents are visible to its waiters
        if (item.y < 0) break;
        const int start = item.x, n = item.y, h = item.z, ib = item.w;
        const int nkb = (n + kTile - 1) / kTile;
        int jlo, jhi;
        near_block_range(ib * kTile, nkb, rsp, rsn, &jlo, &jhi);
        const int nt = jhi - jlo;
        if (nt <= 0) continue;
        for (int t = 0; t < nt; ++t) {
          const int kb = jlo + t;
          int drow = (ib - kb - p.diag_m0) * 128;   // first row of the tile's 256 diagonals
          if (ib - kb - p.diag_m0 < 0 || ib - kb - p.diag_m0 >= p.n_diag) {
            raise_device_error(hdr, DF_ERR_INVALID_ARG, 401);
            drow = 0;
          }
          e_load(&maps.dpk, h, drow, 430);         // C0
          e_load(&maps.dpk, h, drow + 128, 431);   // C1
          if (v_pending) v_load(432);
          // K of the tile, once S of the previous tile (its last reader) is done
          bool ok = !*s_abort;
          if (ok && k_n > 0) ok = wt(k_empty, (k_n - 1) & 1, 433);
          if (ok) {
            load_tile(sK, &maps.k, h * kD, start + kb * kTile, k_full);
            ++k_n;
          }
          e_load(&maps.dpq, h, drow, 434);         // P0
          e_load(&maps.dpq, h, drow + 128, 435);   // P1
          v_head = h;
          v_row = start + kb * kTile;
          v_pending = true;
        }
      }
      if (v_pending) v_load(436);
      // no copy may still be in flight when the CTA leaves
      if (k_n) mbar_wait(k_full, (k_n - 1) & 1, kDrainBudget);
      if (v_n) mbar_wait(v_full, (v_n - 1) & 1, kDrainBudget);
      for (uint32_t b = 0; b < kRing; ++b) {
        if (e_n > b) {
          const uint32_t x = b + kRing * ((e_n - 1 - b) / kRing);  // last load into buffer b
          mbar_wait(e_full + b, (x / kRing) & 1, kDrainBudget);
        }
      }
    }
  } else {
    // ================================================================ compute
    constexpr uint32_t kAll = 0xffffffffu;
    const int g = warp >> 2;             // score columns 32 g .. 32 g + 31
    const int qd = warp & 3;             // TMEM lane quarter
    const int rho = qd * 32 + lane;      // TMEM lane: query row (C, S, O) or key row (P)
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float ks = p.kscale;
    const uint32_t ws = smem_u32(sm + SL::w);
    const uint32_t gW = ws + kRowB * rho + 128u * g;  // this thread's 32 keys of its row
    const int ctid = threadIdx.x;  // 0..511

    auto wait_ph = [&](uint64_t* bar, uint32_t parity, int where) {
      return wait_or_abort(bar, parity, budget, s_abort, hdr, where);
    };

    // Drain one run of a position product from its slot into W (fp32).
    // Columns c = 8 first .. 8 (first + count) - 1 of the slot are diagonals
    // t = 128 half + c.  (Addresses wrap modulo 2^32 where a run starts outside
    // the row; only the stores inside it are made.)
    auto drain = [&](int term, int half, uint32_t slot_col, float kbias) {
      int first, count;
      drain_run(term, half, qd, g, &first, &count);
      const uint32_t src = tmem + slot_col + lane_off + 8u * first;
#pragma unroll 1
      for (int q = 0; q < count; ++q) {
        uint32_t r[8];
        tmem_ld8(src + 8u * q, r);
        tmem_ld_wait(r);
        const int t0 = 128 * half + 8 * (first + q);
        if (term == 0) {
          // C lane rho: diagonal t0 + e goes to key j = rho + 127 - t0 - e of row rho
          const int j0 = rho + 127 - t0;
          st_run_c(ws + kRowB * rho + 4u * (uint32_t)(j0 - 7), r, j0);
        } else {
          // P lane rho (key): diagonal t0 + e goes to row i = t0 + e - 127 + rho, key rho
          const int i0 = t0 - 127 + rho;
          add_run_p(ws + kRowB * (uint32_t)i0 + 4u * rho, r, kbias, i0);
        }
      }
    };
    bool alive = true;

    // The waits of a warp are combined over its lanes (a tensor-memory access
    // is warp-collective: the whole warp issues it or none of it does), and
    // once a wait has failed (the CTA is aborting) the warp arrives on no
    // barrier again.
    uint32_t gt = 0;  // tiles of this CTA so far (each has five products and one P.V)
    // Compute thread 0 takes each work item from the load warp's ring and
    // leaves it in s_cur; the compute warps read it after a barrier of all of
    // them, so that every warp runs the same list.  A failed wait ends the list.
    int4* s_cur = reinterpret_cast<int4*>(sm + SL::next);
    uint32_t ir = 0;  // items taken from the ring (thread 0)
    auto take_item = [&]() {
      const uint32_t slot = ir % kItemRing;
      int4 w = make_int4(-1, -1, -1, -1);
      if (wait_or_abort(item_full + slot, (ir / kItemRing) & 1, budget, s_abort, hdr, 442)) {
        w = s_ring[slot];
        mbar_arrive(item_empty + slot);
      }
      ++ir;
      *s_cur = w;
    };
    // Q rows of an item into tensor memory, the A operand of C0, C1 and S
    // (every MMA that read the previous item's Q is done: this warp waited for
    // that item's last P.V, issued after its last S).  The rows come from
    // global memory whole (warp (qd, g) reads rows 32 qd + 8 g .. + 7, 256 bytes
    // each) into the quarter's rows of W; after the quarter's barrier each lane
    // takes elements 32 g .. 32 g + 31 of its own row into tensor memory, and a
    // second barrier frees the rows for the first C drain.  Rows past the
    // tensor's end are zero.  Nothing for an item without tiles (the MMA warp
    // skips it too).
    auto q_row = [&](const int4& w) { return (long long)w.x + w.w * kTile + rho; };
    auto store_q = [&](const int4& w) {
      if (w.y < 0) return;  // the end of the list
      int lo, hi;
      near_block_range(w.w * kTile, (w.y + kTile - 1) / kTile, rsp, rsn, &lo, &hi);
      if (hi <= lo) return;
      __syncwarp();  // this warp's reads of the same rows (epilogue) are done
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = 32 * qd + 8 * g + 2 * k + (lane >> 4);
        const long long row = (long long)w.x + w.w * kTile + rr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < (long long)p.T)
          v = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + ((size_t)row * p.H + w.z) * kD +
                                              8 * (lane & 15));
        sts128(ws + kRowB * rr + 16 * (lane & 15), v);
      }
      named_sync(2 + qd, 128);  // the quarter's 32 rows are staged
      uint32_t r[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 a = lds128(ws + kRowB * rho + 64 * g + 16 * k);
        r[4 * k] = a.x;
        r[4 * k + 1] = a.y;
        r[4 * k + 2] = a.z;
        r[4 * k + 3] = a.w;
      }
      tmem_st16(tQ + lane_off + 16 * g, r);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (alive && lane == 0) mbar_arrive(q_full);
      named_sync(2 + qd, 128);  // every warp of the quarter has read its Q
    };
    if (ctid == 0) take_item();
    named_sync(1, kComputeThreads);
    for (bool first = true;; first = false) {
      const int4 item = *s_cur;
      if (item.y < 0) break;
      const int start = item.x, n = item.y, h = item.z, i0 = item.w * kTile;
      const int nkb = (n + kTile - 1) / kTile;
      int jlo, jhi;
      near_block_range(i0, nkb, rsp, rsn, &jlo, &jhi);
      const int nt = jhi - jlo;
      if (nt <= 0) {  // (no item of the plan is empty) the item's end, without tiles
        named_sync(1, kComputeThreads);  // every thread has read s_cur
        if (ctid == 0) take_item();
        named_sync(1, kComputeThreads);
        store_q(*s_cur);  // nothing for the end marker or an empty item
        continue;
      }
      if (first) store_q(item);  // later items' Q are stored ahead
      float m_run = -INFINITY, l_run = 0.f;  // l_run: this warp's 32 columns only

      for (int t = 0; t < nt; ++t, ++gt) {
        const uint32_t x0 = 5u * gt;
        // key bias (0, or -inf for a masked or absent key) of this lane's P row,
        // key rho of the tile: the P drains add it to every position term of that
        // key, which masks the key in every score row
        const int jk = (jlo + t) * kTile + rho;
        const float kbias = jk < n ? p.keybias[(size_t)start + jk] : -INFINITY;
        // ---- the four position products in ring order (C0, C1, P0, P1).  C
        // goes into the quarter's rows of W, which are free: the previous
        // tile's reads of them came before the quarter's row-maximum barrier.
        // P is added on top once every row's C is stored.
#pragma unroll 1
        for (int kind = 0; kind < 4; ++kind) {
          if (kind == 2) named_sync(1, kComputeThreads);  // every row's C is stored
          const uint32_t x_k = x0 + kind, s = x_k % kSlots;
          alive = __all_sync(kAll, alive && wait_ph(slot_full + s, (x_k / kSlots) & 1, 450 + kind));
          tc_fence_after();
          if (alive) drain(kind >> 1, kind & 1, s * kSlotCols, kbias);
          tc_fence_before();
          __syncwarp();
          if (alive && lane == 0) mbar_arrive(slot_empty + s);
        }
        if (alive) mbar_arrive(p_drained + qd);  // every lane: its P terms are added
        alive = __all_sync(kAll, alive && wait_ph(p_drained + g, gt & 1, 461));
        float x[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 w4 = lds128(gW + 16u * k);
          x[4 * k + 0] = __uint_as_float(w4.x);
          x[4 * k + 1] = __uint_as_float(w4.y);
          x[4 * k + 2] = __uint_as_float(w4.z);
          x[4 * k + 3] = __uint_as_float(w4.w);
        }
        // ---- S, added to the position terms: raw scores (Q.K + C + P), scaled
        // to log2 units only inside the exponent
        {
          const uint32_t xs = x0 + 4, s = xs % kSlots;
          alive = __all_sync(kAll, alive && wait_ph(slot_full + s, (xs / kSlots) & 1, 462));
          tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[16];
            tmem_ld16(tmem + s * kSlotCols + lane_off + 32 * g + 16 * hf, r);  // whole warp
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 v = add2(make_float2(x[16 * hf + e], x[16 * hf + e + 1]),
                                    make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])));
              x[16 * hf + e] = v.x;
              x[16 * hf + e + 1] = v.y;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (alive && lane == 0) mbar_arrive(slot_empty + s);
        }

        // ---- online softmax (log2 units); row maximum over the four column
        // groups.  The quarter's barrier here also orders this tile's reads of
        // its rows of W before the next tile's C drains into them.
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; e += 2) mt = fmax3(mt, x[e], x[e + 1]);
        mt *= ks;  // log2 units (ks > 0: the maximum commutes with the scaling)
        float* red = sRed + 512 * (gt & 1);
        red[g * 128 + rho] = mt;
        named_sync(2 + qd, 128);  // the four warps of the row quarter
        mt = fmaxf(fmaxf(red[rho], red[128 + rho]), fmaxf(red[256 + rho], red[384 + rho]));
        // Re-base only when the maximum grows by more than 2^8 (exact: numerator and
        // denominator share the stale base).  All four warps of a row agree.
        float scale = 1.f;
        const bool rebase = mt > m_run + 8.f;
        if (rebase) {
          scale = ex2(m_run - mt);
          m_run = mt;
          l_run *= scale;
        }
        // P.V of the previous tile must be done before P is overwritten or O is
        // rescaled
        if (t > 0) alive = __all_sync(kAll, alive && wait_ph(pv_done, (gt - 1) & 1, 463));
        tc_fence_after();
        const float mb = m_run == -INFINITY ? 0.f : m_run;
        {
          uint32_t r[16];
          float2 acc = make_float2(0.f, 0.f);
          const float2 ks2 = make_float2(ks, ks), nmb = make_float2(-mb, -mb);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 arg = fma2(make_float2(x[2 * e], x[2 * e + 1]), ks2, nmb);
            const float p0 = ex2(arg.x);
            const float p1 = ex2(arg.y);
            acc = add2(acc, make_float2(p0, p1));
            r[e] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
          }
          l_run += acc.x + acc.y;
          // keys 32 g .. 32 g + 31 of P: columns 16 g .. 16 g + 15 of the P region
          if (alive) tmem_st16(tP + lane_off + 16 * g, r);
        }
        // O rescaled after P is formed, so that the scores are no longer live
        if (alive && t > 0 && __any_sync(kAll, rebase)) {
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[16];
            tmem_ld16(tO + lane_off + 32 * g + 16 * hf, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
            tmem_st16(tO + lane_off + 32 * g + 16 * hf, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (alive && lane == 0) mbar_arrive(p_full);
      }

      // the next item, taken while the tiles ran; read after this barrier (every
      // thread read the current one before its first tile)
      if (ctid == 0) take_item();
      named_sync(1, kComputeThreads);
      // the next item's Q rows (two 128-byte lines each) into L1 while the
      // epilogue runs
      {
        const int4 nx = *s_cur;
        const long long row = q_row(nx);
        if (nx.y >= 0 && row < (long long)p.T)
          asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const T*>(p.q) +
                                                        ((size_t)row * p.H + nx.z) * kD + 32 * g));
      }
      // ---- epilogue: final rows, or the partial state for the far-tile kernel
      alive = __all_sync(kAll, alive && wait_ph(pv_done, (gt - 1) & 1, 464));
      tc_fence_after();
      float* red = sRed + 1024;
      red[g * 128 + rho] = l_run;
      named_sync(2 + qd, 128);
      const float l_tot = (red[rho] + red[128 + rho]) + (red[256 + rho] + red[384 + rho]);
      const bool store = alive && *s_abort == 0;
      const bool has_far = jlo > 0 || jhi < nkb;
      // O (divided by the row sum for final rows) goes through the quarter's
      // rows of W, so that the stores to global memory are whole rows: after
      // the quarter's barrier each warp writes 8 rows of its quarter.
      {
        const float sc = has_far ? 1.f : (l_tot > 0.f ? 1.f / l_tot : 0.f);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[8];
          tmem_ld8(tO + lane_off + 32 * g + 8 * c, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 8; e += 4)
            sts128(ws + kRowB * rho + 128 * g + 32 * c + 4 * e,
                   make_uint4(__float_as_uint(__uint_as_float(r[e]) * sc),
                              __float_as_uint(__uint_as_float(r[e + 1]) * sc),
                              __float_as_uint(__uint_as_float(r[e + 2]) * sc),
                              __float_as_uint(__uint_as_float(r[e + 3]) * sc)));
        }
      }
      if (has_far && g == 0 && store && i0 + rho < n)
        partial_ml(p)[((size_t)start + i0 + rho) * p.H + h] = make_float2(m_run, l_tot);
      named_sync(2 + qd, 128);  // the quarter's 32 rows are staged
      if (store) {
        if (has_far) {
          // un-normalised fp32 rows (512 bytes): one row per pass of the warp
#pragma unroll 2
          for (int k = 0; k < 8; ++k) {
            const int rr = 32 * qd + 8 * g + k;
            const uint4 v = lds128(ws + kRowB * rr + 16 * lane);
            if (i0 + rr < n)
              *reinterpret_cast<uint4*>(partial_o(p) + ((size_t)start + i0 + rr) * p.H * kD + h * kD +
                                        4 * lane) = v;
          }
        } else {
          // final rows in the I/O type (256 bytes): lanes 16 a .. 16 a + 15 one row
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 32 * qd + 8 * g + 2 * k + (lane >> 4);
            const uint32_t a = ws + kRowB * rr + 32 * (lane & 15);
            const uint4 v0 = lds128(a), v1 = lds128(a + 16);
            const size_t tok = (size_t)start + i0 + rr;
            if (i0 + rr < n && p.keybias[tok] == 0.f) {
              uint4 w;
              w.x = BF16 ? pack_bf16x2(__uint_as_float(v0.x), __uint_as_float(v0.y))
                         : pack_f16x2(__uint_as_float(v0.x), __uint_as_float(v0.y));
              w.y = BF16 ? pack_bf16x2(__uint_as_float(v0.z), __uint_as_float(v0.w))
                         : pack_f16x2(__uint_as_float(v0.z), __uint_as_float(v0.w));
              w.z = BF16 ? pack_bf16x2(__uint_as_float(v1.x), __uint_as_float(v1.y))
                         : pack_f16x2(__uint_as_float(v1.x), __uint_as_float(v1.y));
              w.w = BF16 ? pack_bf16x2(__uint_as_float(v1.z), __uint_as_float(v1.w))
                         : pack_f16x2(__uint_as_float(v1.z), __uint_as_float(v1.w));
              *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (tok * p.H + h) * kD + 8 * (lane & 15)) = w;
            }
          }
        }
      }
      // the next item's Q (its rows were prefetched into L1 before the
      // epilogue; s_cur holds the item until the end of its tiles)
      store_q(*s_cur);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kComputeWarps) tmem_dealloc(tmem, 512);
}

int near_sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

template <bool BF16>
cudaError_t launch_typed(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(tc_near128_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Smem::bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.max_items, near_sm_count());
  e = launch_after_plan(tc_near128_kernel<BF16>, grid, kThreads, Smem::bytes, s, p, maps);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_near128(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  return p.dtype == DF_BF16 ? launch_typed<true>(p, maps, s) : launch_typed<false>(p, maps, s);
}

}  // namespace dfa
