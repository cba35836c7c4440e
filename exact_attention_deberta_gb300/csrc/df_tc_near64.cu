// Near-tile fused forward for head size 64 on tcgen05 (bf16 / fp16 I/O; fp32
// accumulation and fp32 position terms).
//
// Operation: DisentangledFlash README "Status" (C2P/P2C disentangled attention,
// FP16/BF16, packed cu_seqlens) and the kernels-community "DisentangledFlash"
// discussion "Motivation" (exact, tiled and streaming, no [B,H,L,L] matrix).
//
// Diagonal form of the position terms.  In a 128 x 128 tile with query block
// i0 and key block j0 = i0 - 128 m, element (i', j') has relative distance
// r = 128 m - 127 + t with t = i' - j' + 127, the tile's diagonal (0..254).
// The planning kernel stores, per offset m, the PK and PQ rows at idx(r) for
// every diagonal (the diagonal tables), so that MMAs give
//     C[i'][t] = Q_i . PK[idx(r_t)]      P[j'][t] = K_j . PQ[idx(r_t)]
// and the score element needs C[i'][i' - j' + 127] + P[j'][i' - j' + 127]: a
// fixed skew, with no index lookups.  Each term comes in two halves of 128
// diagonals (t < 128, t >= 128): four position products per tile (C0, P0, C1,
// P1), each a 128 x 128 x 64 MMA.
//
// Skew through shared memory, in fp32.  Both terms are stored by query row,
// in the order the score row reads them:
//     Cw[i'][j'] = C[i'][i' - j' + 127]      Pw[i'][j'] = P[j'][i' - j' + 127]
// A lane of C (query row i') writes its diagonals t into its own row at key
// i' + 127 - t; a lane of P (key row j') writes diagonal t into query row
// t - 127 + j' at key j'.  Rows are 132 words (528 bytes): the 32 lanes of a
// drain store land in 32 different banks (word 133 i' + const, 133 being odd)
// and the gather reads a row's 32 keys as 16-byte vectors without conflicts
// (rows 33 sixteen-byte units apart).  A lane quarter needs 160 of the 256
// diagonals of either term; each of its four warps drains one contiguous run of
// 8-column groups per product (balanced: 10 groups per warp per tile).
//
// Tensor memory: a ring of three 128-column slots takes the products in the
// order C0, P0, C1, P1, S of every tile (product x in slot x mod 3), so that
// the tensor core computes the next products while the current ones are
// drained; P (16-bit pairs, for P.V) overwrites its tile's S; O 384-447; Q
// (16-bit pairs, the A operand of C0, C1 and S) 448-479; when the kernel forms
// the far tiles' query scalars and key terms (p.scal_in_near), Q and the
// diagonal tile's K times the head's selector rows in 480-495 and 496-511.
//
// Roles (one CTA per SM, persistent over the work list):
//   warps 0-15  compute: warp w owns TMEM lanes 32 (w % 4) .. +31 (query rows
//               for C, S and O; key rows for P) and score columns
//               32 (w / 4) .. +31 of every tile; they drain the position
//               products, gather, run the online softmax, write P into TMEM
//               and store each item's Q rows into TMEM;
//   warp 16     MMA issue (one thread): every tcgen05.mma;
//   warp 17     TMA loads (one thread): K, V and the diagonal-table halves
//               through a three-buffer ring; it also claims the work items
//               (longest first, one global counter) and hands them to the
//               other roles.
// No barrier of the whole CTA inside a tile: the compute warps hand the skew
// buffers over by lane quarter.  Quarter q's drains fill the rows 32 q .. +31
// of Cw and the key columns 32 q .. +31 of Pw; a warp gathers from its own
// quarter's rows and its column group's keys, so it waits for those two
// quarters' drains only, and a quarter drains the next tile once the gathers
// that read its rows and its columns are done.  The row maximum and sum are
// exchanged between the four warps of a row quarter only.
// A masked or absent key is masked through its P row: the P drains add the
// key's bias (0 or -inf) to every position term they store for it.
// The kernel does not spill (ptxas: 96 registers, no local memory), so no
// destination register of an asynchronous tensor-memory load is spilled or
// reused before its wait.
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

constexpr int kD = 64;
constexpr int kTile = 128;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 64;  // + the MMA warp and the load warp
constexpr uint32_t kRowW = 132;           // words per Cw / Pw row: 128 keys + 4 of padding
constexpr uint32_t kRowB = kRowW * 4;     // 528 bytes
static_assert((kRowW + 1) % 2 == 1 && (kRowB / 16) % 2 == 1, "conflict-free drains and gathers");

// Tensor-memory columns.
constexpr uint32_t kSlots = 3, kSlotCols = 128;
constexpr uint32_t kColO = kSlots * kSlotCols;  // 384
constexpr uint32_t kColQ = kColO + kD;          // 448: Q (16-bit pairs), the A operand of C0, C1, S
static_assert(tmem_region_fits(0, kSlots * kSlotCols, kColO), "product ring below O");
static_assert(tmem_region_fits(kColO, kD, kColQ), "O below Q");
static_assert(tmem_region_fits(kColQ, kD / 2, 512), "Q inside 512 columns");
// The far tiles' per-token terms, when this kernel forms them: Q.[PK|PQ rows]
// (16 columns, the query scalars in the first two) and K.[PK|PQ rows] of the
// diagonal tile's keys (16 columns, the key terms in columns 2 and 3)
constexpr uint32_t kColAB = kColQ + kD / 2;     // 480
static_assert(tmem_region_fits(kColAB, 32, 512), "scalar products inside 512 columns");
constexpr uint32_t kSelBytes = 16 * kD * 2;     // one head's 16 selector rows
// P of a tile (16-bit pairs) overwrites its S: column group c's 32 keys at
// columns 32 c .. 32 c + 15 of the S slot
static_assert(32 * (kTile / 32 - 1) + 16 <= kSlotCols, "P inside the S slot");
constexpr uint32_t kRing = 3;                   // diagonal-table halves in flight
constexpr uint32_t kItemRing = 4;               // work items handed from the load warp to the others

struct Smem {
  static constexpr uint32_t k = 0;                     // K tile
  static constexpr uint32_t v = k + kBoxBytes;         // V tile
  static constexpr uint32_t e = v + kBoxBytes;         // [kRing] diagonal-table halves
  static constexpr uint32_t sel = e + kRing * kBoxBytes;  // [2] selector rows (by item parity)
  static constexpr uint32_t cw = sel + 2 * kSelBytes;  // fp32 [128][132]
  static constexpr uint32_t pw = cw + 128 * kRowB;     // fp32 [128][132]
  static constexpr uint32_t red = pw + 128 * kRowB;    // float [3][4][128]: row max / sum exchange
  static constexpr uint32_t bars = red + 3 * 4 * 128 * 4;
  static constexpr int kBars = 36 + 2 * kItemRing;
  static constexpr uint32_t misc = bars + kBars * 8;   // abort flag, TMEM slot
  static constexpr uint32_t next = (misc + 16 + 15) & ~15u;  // int4: the compute warps' next item
  static constexpr uint32_t ring = next + 16;                // int4 [kItemRing]: items handed out
  static constexpr uint32_t bytes = ring + 16 * kItemRing;
};
// 16-byte vector accesses: the next item (int4) and the skew buffers' rows
static_assert(Smem::next % 16 == 0 && Smem::ring % 16 == 0 && Smem::cw % 16 == 0 &&
                  Smem::pw % 16 == 0,
              "16-byte aligned vector regions");
static_assert(Smem::bytes <= 227 * 1024, "near-tile shared memory");
static_assert(Smem::bars % 8 == 0 && Smem::e % 1024 == 0 && Smem::sel % 1024 == 0, "alignment");

// Run of 8-column groups (first group, count) that warp g of lane quarter qd
// drains from position product `kind` (0: C0, 1: P0, 2: C1, 3: P1).  Lane quarter
// qd needs diagonals [32 qd, 32 qd + 159] of C and [96 - 32 qd, 255 - 32 qd] of P;
// each product's groups are split into four equal runs.
__device__ __forceinline__ void drain_run(int kind, int qd, int g, int* first, int* count) {
  int lo, len;
  switch (kind) {
    case 0: lo = 4 * qd; len = 4 - qd; break;           // C, t in [32 qd, 128)
    case 1: lo = 12 - 4 * qd; len = 1 + qd; break;      // P, t in [96 - 32 qd, 128)
    case 2: lo = 0; len = qd + 1; break;                 // C, t in [128, 160 + 32 qd)
    default: lo = 0; len = 4 - qd; break;                // P, t in [128, 256 - 32 qd)
  }
  *first = lo + g * len;
  *count = len;
}

// Skew stores of one 8-diagonal run, each made only when its key (row) lies
// in 0 .. 127.  C: value e to key j0 - e of the lane's row, i.e. byte offset
// 4 (7 - e) from the run's lowest key (a7); P: value e to row i0 + e of the
// lane's key column (offset kRowB e from a0).  The base addresses stay inside
// the shared window even where a run starts outside the tile.
__device__ __forceinline__ void st_run_c(uint32_t a7, const uint32_t* r, int j0) {
#define DFA_C(e) sts32_below_at<4 * (7 - e)>(a7, r[e], (uint32_t)(j0 - (e)), 128u);
  DFA_C(0) DFA_C(1) DFA_C(2) DFA_C(3) DFA_C(4) DFA_C(5) DFA_C(6) DFA_C(7)
#undef DFA_C
}
__device__ __forceinline__ void st_run_p(uint32_t a0, const uint32_t* v, int i0) {
#define DFA_P(e) sts32_below_at<(int)kRowB * e>(a0, v[e], (uint32_t)(i0 + (e)), 128u);
  DFA_P(0) DFA_P(1) DFA_P(2) DFA_P(3) DFA_P(4) DFA_P(5) DFA_P(6) DFA_P(7)
#undef DFA_P
}

// Bits of a 16-bit value, for packing two of them into a 32-bit word.
__device__ __forceinline__ uint16_t bits16(__nv_bfloat16 v) { return __bfloat16_as_ushort(v); }
__device__ __forceinline__ uint16_t bits16(__half v) { return __half_as_ushort(v); }

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_near64_kernel(const Problem p, const __grid_constant__ TcMaps maps) {
  using SL = Smem;
  constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, kD, BF16 ? 1 : 0, 0, 1);
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    grid_dependency_wait();
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(p.hdr, DF_ERR_CUDA, 260);
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
  uint64_t* e_empty = bars + 7;     // [kRing] the product that read the half is done
  uint64_t* slot_full = bars + 10;  // [3] product in the slot computed
  uint64_t* slot_empty = bars + 13; // [3] product drained (one arrival per compute warp)
  uint64_t* p_full = bars + 16;     // P of the tile in TMEM (one arrival per compute warp)
  uint64_t* pv_done = bars + 17;    // P.V of the tile done (O, P and V free)
  uint64_t* bar_end = bars + 18;    // every MMA done (exit)
  // Tile hand-offs between compute warps, by lane quarter q (rows 32 q .. +31,
  // keys 32 q .. +31): the quarter's drains are stored (its C rows and P
  // columns); the gathers of the quarter's rows are done; the gathers of its
  // key columns are done.  One phase per tile; every thread of the four
  // contributing warps arrives.
  uint64_t* drained = bars + 19;    // [4]
  uint64_t* row_read = bars + 23;   // [4]
  uint64_t* col_read = bars + 27;   // [4]
  // Work items: the load warp takes the next item of the list (a global
  // counter, longest items first) and hands it to the MMA warp and the compute
  // warps through a ring of kItemRing slots; a slot is free again once both
  // have read it.  An item with n < 0 ends the CTA's list.
  uint64_t* item_full = bars + 31;  // [kItemRing]
  uint64_t* item_empty = bars + 31 + kItemRing;  // [kItemRing] (MMA thread and compute thread 0)
  // Far tiles' terms (when p.scal_in_near): an item's selector rows landed
  // (by item parity); the MMAs that read them are done; both products of the
  // item are in tensor memory.
  uint64_t* sel_full = bars + 31 + 2 * kItemRing;   // [2]
  uint64_t* sel_empty = sel_full + 2;               // [2]
  uint64_t* ab_full = sel_full + 4;
  uint8_t* sSel = sm + SL::sel;
  int4* s_ring = reinterpret_cast<int4*>(sm + SL::ring);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SL::misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < SL::kBars; ++b) mbar_init(bars + b, 1);
    for (int s = 0; s < 3; ++s) mbar_init(slot_empty + s, kComputeWarps);
    mbar_init(p_full, kComputeWarps);
    mbar_init(q_full, kComputeWarps);
    for (uint32_t s = 0; s < kItemRing; ++s) mbar_init(item_empty + s, 2);
    for (int q = 0; q < 4; ++q) {
      mbar_init(drained + q, 128);
      mbar_init(row_read + q, 128);
      mbar_init(col_read + q, 128);
    }
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
  const uint32_t tO = tmem + kColO, tQ = tmem + kColQ;

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
      uint32_t ec_n = 0, pp = 0, pv_n = 0, k_n = 0, v_n = 0, q_n = 0, g_n = 0, ia = 0;
      constexpr uint32_t kIdescAB = idesc_f16(128, 16, BF16 ? 1 : 0, 0, 0);
      bool have_prev = false, prev_first = false;
      const uint64_t dk = kmajor_desc(sK, 0);
      const uint32_t dv_addr = smem_u32(sV);

      // Position product `kind` (0 C0, 1 P0, 2 C1, 3 P1) into the next ring slot:
      // C = Q.table (Q from tensor memory), P = K.table.
      auto issue_pos = [&](int kind, int where) {
        const uint32_t x = pp, s = x % 3, b = ec_n % kRing;
        bool ok = !*s_abort;
        if (ok && x >= 3) ok = wt(slot_empty + s, ((x / 3) - 1) & 1, where);
        // C1 takes the slot of the previous tile's S, where P lived until its
        // P.V was done
        if (ok && kind == 2 && g_n > 0) ok = wt(pv_done, (g_n - 1) & 1, where + 2);
        ok = wt(e_full + b, (ec_n / kRing) & 1, where + 1) && ok;
        if (!ok) return;
        tc_fence_after();
        const uint64_t db = kmajor_desc(sE + b * kBoxBytes, 0);
        const uint32_t d = tmem + s * kSlotCols;
        if (kind & 1) {
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
      // O (+)= P.V of the previous tile; P is in that tile's S slot, warp
      // column group c at columns 32 c .. 32 c + 15 (16-bit pairs).
      auto issue_pv = [&](bool first, int where) {
        bool ok = wt(p_full, pv_n & 1, where);
        ok = wt(v_full, v_n & 1, where + 1) && ok;
        if (!ok) return;
        ++v_n;
        tc_fence_after();
        const uint32_t ps = tmem + ((5u * pv_n + 4u) % 3u) * kSlotCols;
        const uint64_t dv = vtile_desc(dv_addr, 0);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_ts(tO, ps + 32 * (k >> 1) + 8 * (k & 1), dv + vtile_step(k), kIdescPV,
                 (!first || k > 0) ? 1u : 0u);
        mma_commit(pv_done);
        ++pv_n;
      };

      for (uint32_t ic = 0;; ++ic) {
        const uint32_t slot = ic % kItemRing;
        if (!wt(item_full + slot, (ic / kItemRing) & 1, 341)) break;
        const int4 item = s_ring[slot];
        mbar_arrive(item_empty + slot);
        if (item.y < 0) break;
        const int n = item.y, ib = item.w;
        const int nkb = (n + kTile - 1) / kTile;
        int jlo, jhi;
        near_block_range(ib * kTile, nkb, rsp, rsn, &jlo, &jhi);
        const int nt = jhi - jlo;
        if (nt <= 0) continue;
        const int t_diag = ib - jlo;  // the diagonal tile (never saturated)
        const uint64_t dsel = kmajor_desc(sSel + (ia & 1) * kSelBytes, 0);
        for (int t = 0; t < nt; ++t) {
          // The previous tile's P.V goes first at an item's first tile: the
          // compute warps store this item's Q once that P.V is done.
          if (t == 0) {
            if (have_prev) issue_pv(prev_first, 320);
            wt(q_full, q_n & 1, 304);
            ++q_n;
            // the query rows' far-tile scalars: Q.[PK|PQ rows]
            if (p.scal_in_near && !*s_abort && wt(sel_full + (ia & 1), (ia >> 1) & 1, 324)) {
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < kD / 16; ++k)
                mma_ts(tmem + kColAB, tQ + 8 * k, dsel + kmajor_step(k), kIdescAB, k > 0 ? 1u : 0u);
            }
          }
          issue_pos(0, 310);
          wt(k_full, k_n & 1, 305);
          ++k_n;
          // the diagonal tile's keys: K.[PK|PQ rows], the far tiles' key terms
          if (p.scal_in_near && t == t_diag) {
            if (!*s_abort) {
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < kD / 16; ++k)
                mma_ss(tmem + kColAB + 16, dk + kmajor_step(k), dsel + kmajor_step(k), kIdescAB, k > 0);
            }
            mma_commit(ab_full);
            mma_commit(sel_empty + (ia & 1));
            ++ia;
          }
          issue_pos(1, 312);
          if (t > 0) issue_pv(prev_first, 320);
          issue_pos(2, 314);
          issue_pos(3, 316);
          // S = Q.K^T into the next slot
          {
            const uint32_t x = pp, s = x % 3;
            bool ok = !*s_abort;
            if (ok && x >= 3) ok = wt(slot_empty + s, ((x / 3) - 1) & 1, 318);
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
          ++g_n;
          have_prev = true;
          prev_first = t == 0;
        }
      }
      if (have_prev) issue_pv(prev_first, 322);
      // no MMA may still be in flight when the CTA leaves
      mma_commit(bar_end);
      mbar_wait(bar_end, 0, kDrainBudget);
    }
  } else if (warp == kComputeWarps + 1) {
    // ================================================================ loads
    // One thread issues every TMA load, in the order in which the MMAs free
    // the buffers (C0, P0, C1, P1 of a tile through a ring of kRing table
    // buffers; K once the previous S is done; V one tile late, once the P.V
    // before it is done), so that no load waits behind another's condition.
    if (lane == 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dpk);
      tma_prefetch_desc(&maps.dpq);
      if (p.scal_in_near) tma_prefetch_desc(&maps.absel);
      uint32_t k_n = 0, v_n = 0, e_n = 0, ia = 0;
      int v_head = 0, v_row = 0;
      bool v_pending = false;
      auto e_load = [&](const CUtensorMap* map, int head, int row, int where) {
        const uint32_t b = e_n % kRing;
        bool ok = !*s_abort;
        if (ok && e_n >= kRing) ok = wt(e_empty + b, ((e_n / kRing) - 1) & 1, where);
        if (ok) {
          mbar_expect_tx(e_full + b, kBoxBytes);
          tma_load_2d(sE + b * kBoxBytes, map, head * kD, row, e_full + b);
          ++e_n;
        }
      };
      // V of the previous tile, once the P.V before it is done
      auto v_load = [&](int where) {
        bool ok = !*s_abort;
        if (ok && v_n > 0) ok = wt(pv_done, (v_n - 1) & 1, where);
        if (ok) {
          mbar_expect_tx(v_full, kBoxBytes);
          tma_load_2d(sV, &maps.v, v_head * kD, v_row, v_full);
          ++v_n;
        }
        v_pending = false;
      };
      for (uint32_t ic = 0;; ++ic) {
        // the next item of the list, claimed once its ring slot is free and
        // handed to the other roles
        const uint32_t slot = ic % kItemRing;
        if (ic >= kItemRing && !wt(item_empty + slot, ((ic / kItemRing) - 1) & 1, 340)) break;
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
        // the head's selector rows, into the buffer of this item's parity once
        // the MMAs of the item two back are done with it
        if (p.scal_in_near) {
          const uint32_t sb = ia & 1;
          bool ok = !*s_abort;
          if (ok && ia >= 2) ok = wt(sel_empty + sb, ((ia >> 1) - 1) & 1, 343);
          if (ok) {
            mbar_expect_tx(sel_full + sb, kSelBytes);
            tma_load_2d(sSel + sb * kSelBytes, &maps.absel, 0, h * 16, sel_full + sb);
          }
          ++ia;
        }
        for (int t = 0; t < nt; ++t) {
          const int kb = jlo + t;
          int drow = (ib - kb - p.diag_m0) * 128;   // first row of the tile's 256 diagonals
          if (ib - kb - p.diag_m0 < 0 || ib - kb - p.diag_m0 >= p.n_diag) {
            raise_device_error(hdr, DF_ERR_INVALID_ARG, 261);
            drow = 0;
          }
          e_load(&maps.dpk, h, drow, 301);              // C0
          e_load(&maps.dpq, h, drow, 302);              // P0
          if (v_pending) v_load(308);
          e_load(&maps.dpk, h, drow + 128, 306);        // C1
          // K of the tile, once S of the previous tile (its last reader) is done
          bool ok = !*s_abort;
          if (ok && k_n > 0) ok = wt(k_empty, (k_n - 1) & 1, 303);
          if (ok) {
            mbar_expect_tx(k_full, kBoxBytes);
            tma_load_2d(sK, &maps.k, h * kD, start + kb * kTile, k_full);
            ++k_n;
          }
          e_load(&maps.dpq, h, drow + 128, 307);        // P1
          v_head = h;
          v_row = start + kb * kTile;
          v_pending = true;
        }
      }
      if (v_pending) v_load(309);
      // no copy may still be in flight when the CTA leaves
      if (k_n) mbar_wait(k_full, (k_n - 1) & 1, kDrainBudget);
      if (v_n) mbar_wait(v_full, (v_n - 1) & 1, kDrainBudget);
      for (uint32_t x = ia > 2 ? ia - 2 : 0; x < ia; ++x) mbar_wait(sel_full + (x & 1), (x >> 1) & 1, kDrainBudget);
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
    const uint32_t cw = smem_u32(sm + SL::cw), pw = smem_u32(sm + SL::pw);
    const uint32_t gC = cw + kRowB * rho + 128u * g, gP = pw + kRowB * rho + 128u * g;
    const int ctid = threadIdx.x;  // 0..511

    auto wait_ph = [&](uint64_t* bar, uint32_t parity, int where) {
      return wait_or_abort(bar, parity, budget, s_abort, hdr, where);
    };

    // Drain one run of a position product from its slot into Cw / Pw (fp32).
    // Columns c = 8 first .. 8 (first + count) - 1 of the slot are diagonals
    // t = 128 half + c.
    // (Addresses wrap modulo 2^32 where a run starts outside the row; only the
    // stores inside it are made.)
    auto store_run = [&](int kind, int first, const uint32_t* r, float kbias) {
      const int t0 = 128 * (kind >> 1) + 8 * first;
      if ((kind & 1) == 0) {
        // C lane rho: diagonal t0 + e goes to key j = rho + 127 - t0 - e of row rho
        // (addresses from the lowest key of the run, j0 - 7)
        const int j0 = rho + 127 - t0;
        const uint32_t a7 = cw + kRowB * rho + 4u * (uint32_t)(j0 - 7);
        st_run_c(a7, r, j0);
      } else {
        // P lane rho (key): diagonal t0 + e goes to row i = t0 + e - 127 + rho, key rho
        const int i0 = t0 - 127 + rho;
        const uint32_t a0 = pw + kRowB * (uint32_t)i0 + 4u * rho;
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(__uint_as_float(r[e]) + kbias);
        st_run_p(a0, v, i0);
      }
    };
    auto drain = [&](int kind, uint32_t slot_col, float kbias) {
      int first, count;
      drain_run(kind, qd, g, &first, &count);
      const uint32_t src = tmem + slot_col + lane_off + 8u * first;
#pragma unroll 1
      for (int q = 0; q < count; ++q) {
        uint32_t r[8];
        tmem_ld8(src + 8u * q, r);
        tmem_ld_wait(r);
        store_run(kind, first + q, r, kbias);
      }
    };

    // The waits of a warp are combined over its lanes (a tensor-memory access
    // is warp-collective: the whole warp issues it or none of it does), and
    // once a wait has failed (the CTA is aborting) the warp arrives on no
    // barrier again.
    bool alive = true;
    uint32_t gt = 0;  // tiles of this CTA so far (each has five products and one P.V)
    uint32_t ia = 0;  // items whose far-tile terms were formed (p.scal_in_near)
    // Compute thread 0 takes each work item from the load warp's ring and
    // leaves it in s_cur; the compute warps read it after a barrier of all of
    // them, so that every warp runs the same list.  A failed wait ends the list.
    int4* s_cur = reinterpret_cast<int4*>(sm + SL::next);
    uint32_t ir = 0;  // items taken from the ring (thread 0)
    auto take_item = [&]() {
      const uint32_t slot = ir % kItemRing;
      int4 w = make_int4(-1, -1, -1, -1);
      if (wait_or_abort(item_full + slot, (ir / kItemRing) & 1, budget, s_abort, hdr, 342)) {
        w = s_ring[slot];
        mbar_arrive(item_empty + slot);
      }
      ++ir;
      *s_cur = w;
    };
    // Q rows of an item into tensor memory, the A operand of C0, C1 and S
    // (every MMA that read the previous item's Q is done: this warp waited for
    // that item's last S).  The rows come from global memory whole (warp
    // (qd, g) reads rows 32 qd + 8 g .. + 7, 128 bytes each) into the idle Pw
    // buffer; after the quarter's barrier each lane takes columns 8 g .. 8 g + 7
    // (elements 16 g .. 16 g + 15) of its own row into tensor memory.  Rows past
    // the tensor's end are zero.  Nothing for an item without tiles (the MMA
    // warp skips it too).
    auto q_row = [&](const int4& w) { return (long long)w.x + w.w * kTile + rho; };
    const uint32_t qs = smem_u32(sm + SL::pw);
    auto store_q = [&](const int4& w) {
      if (w.y < 0) return;  // the end of the list
      int lo, hi;
      near_block_range(w.w * kTile, (w.y + kTile - 1) / kTile, rsp, rsn, &lo, &hi);
      if (hi <= lo) return;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int rr = 32 * qd + 8 * g + 4 * k + (lane >> 3);
        const long long row = (long long)w.x + w.w * kTile + rr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < (long long)p.T)
          v = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + ((size_t)row * p.H + w.z) * kD +
                                              8 * (lane & 7));
        sts128(qs + kRowB * rr + 16 * (lane & 7), v);
      }
      named_sync(2 + qd, 128);  // the quarter's 32 rows are staged
      const uint4 a0 = lds128(qs + kRowB * rho + 32 * g), a1 = lds128(qs + kRowB * rho + 32 * g + 16);
      const uint32_t r[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      tmem_st8(tQ + lane_off + 8 * g, r);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (alive && lane == 0) mbar_arrive(q_full);
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
        // the quarter's C rows and P columns are free once the previous tile's
        // gathers that read them are done
        if (gt > 0)
          alive = __all_sync(kAll, alive && wait_ph(row_read + qd, (gt - 1) & 1, 288) &&
                                       wait_ph(col_read + qd, (gt - 1) & 1, 289));
        // ---- the four position products, drained in ring order
#pragma unroll 1
        for (int kind = 0; kind < 4; ++kind) {
          const uint32_t x = x0 + kind, s = x % 3;
          alive = __all_sync(kAll, alive && wait_ph(slot_full + s, (x / 3) & 1, 290 + kind));
          tc_fence_after();
          if (alive) drain(kind, s * kSlotCols, kbias);
          tc_fence_before();
          __syncwarp();
          if (alive && lane == 0) mbar_arrive(slot_empty + s);
        }
        if (alive) mbar_arrive(drained + qd);  // every lane: its stores are published
        // ---- S, then the position terms of this thread's 32 elements: raw
        // scores (Q.K + C + P), scaled to log2 units only inside the exponent
        float x[32];
        {
          const uint32_t xs = x0 + 4, s = xs % 3;
          alive = __all_sync(kAll, alive && wait_ph(slot_full + s, (xs / 3) & 1, 294));
          tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[16];
            tmem_ld16(tmem + s * kSlotCols + lane_off + 32 * g + 16 * hf, r);  // whole warp
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 16; ++e) x[16 * hf + e] = __uint_as_float(r[e]);
          }
          tc_fence_before();
          __syncwarp();
          if (alive && lane == 0) mbar_arrive(slot_empty + s);
        }
        // the C row of this thread (quarter qd) and the P columns of its keys
        // (quarter g) are stored
        alive = __all_sync(kAll, alive && wait_ph(drained + qd, gt & 1, 297) &&
                                     (g == qd || wait_ph(drained + g, gt & 1, 298)));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 c4 = lds128(gC + 16u * k), p4 = lds128(gP + 16u * k);
          const float2 a = add2(make_float2(__uint_as_float(c4.x), __uint_as_float(c4.y)),
                                make_float2(__uint_as_float(p4.x), __uint_as_float(p4.y)));
          const float2 b = add2(make_float2(__uint_as_float(c4.z), __uint_as_float(c4.w)),
                                make_float2(__uint_as_float(p4.z), __uint_as_float(p4.w)));
          const float2 s0 = add2(make_float2(x[4 * k + 0], x[4 * k + 1]), a);
          const float2 s1 = add2(make_float2(x[4 * k + 2], x[4 * k + 3]), b);
          x[4 * k + 0] = s0.x;
          x[4 * k + 1] = s0.y;
          x[4 * k + 2] = s1.x;
          x[4 * k + 3] = s1.y;
        }

        // ---- online softmax (log2 units); row maximum over the four column groups
        if (alive) {  // every lane: its reads of Cw row rho and Pw columns 32 g .. +31 are done
          mbar_arrive(row_read + qd);
          mbar_arrive(col_read + g);
        }
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
        // P.V of the previous tile must be done before O is rescaled or P is overwritten
        if (t > 0) alive = __all_sync(kAll, alive && wait_ph(pv_done, (gt - 1) & 1, 295));
        tc_fence_after();
        if (alive && t > 0 && __any_sync(kAll, rebase)) {
          uint32_t r[16];
          tmem_ld16(tO + lane_off + 16 * g, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
          tmem_st16(tO + lane_off + 16 * g, r);
        }
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
          // P over this warp's own S columns (read above by this warp only)
          if (alive) tmem_st16(tmem + ((x0 + 4u) % 3u) * kSlotCols + lane_off + 32 * g, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (alive && lane == 0) mbar_arrive(p_full);
        // ---- after the diagonal tile: the far tiles' terms of this query block
        // (query scalars, log2-scaled) and of its keys (raw key terms as
        // hi + lo, masked keys at the finite stand-in), one warp per quarter
        if (p.scal_in_near && t == item.w - jlo) {
          if (g == 0) {
            alive = __all_sync(kAll, alive && wait_ph(ab_full, ia & 1, 299));
            tc_fence_after();
            if (alive) {
              uint32_t ra[8], rb[8];
              tmem_ld8(tmem + kColAB + lane_off, ra);
              tmem_ld8(tmem + kColAB + 16 + lane_off, rb);
              tmem_ld_wait(ra);
              tmem_ld_wait(rb);
              const int i = i0 + rho;  // query row; also key row of the diagonal tile
              if (i < n) {
                const size_t tok = (size_t)start + i;
                float* sc = p.scal + (size_t)h * 4 * p.t_pad + tok;
                sc[0] = __uint_as_float(ra[0]) * ks;
                sc[p.t_pad] = __uint_as_float(ra[1]) * ks;
                const bool valid = kbias == 0.f;
                const float c0 = valid ? __uint_as_float(rb[2]) : kMaskedKeyTerm;
                const float c1 = valid ? __uint_as_float(rb[3]) : kMaskedKeyTerm;
                const T h0 = IO<T>::from_f(c0), h1 = IO<T>::from_f(c1);
                const T l0 = IO<T>::from_f(valid ? c0 - IO<T>::to_f(h0) : kMaskedKeyTerm);
                const T l1 = IO<T>::from_f(valid ? c1 - IO<T>::to_f(h1) : kMaskedKeyTerm);
                uint4 w0;
                w0.x = (uint32_t)bits16(h0) | ((uint32_t)bits16(l0) << 16);
                w0.y = (uint32_t)bits16(h1) | ((uint32_t)bits16(l1) << 16);
                w0.z = 0u;
                w0.w = 0u;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.kaug) + (tok * p.H + h) * 16);
                dst[0] = w0;
                dst[1] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
            tc_fence_before();
          }
          ++ia;
        }
      }

      // the next item, taken while the tiles ran; read after this barrier (every
      // thread read the current one before its first tile)
      if (ctid == 0) take_item();
      named_sync(1, kComputeThreads);
      const int4 nx = *s_cur;
      // the next item's Q rows (one 128-byte line each) into L1 while the
      // epilogue runs
      if (nx.y >= 0) {
        const long long row = q_row(nx);
        if (row < (long long)p.T)
          asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const T*>(p.q) +
                                                        ((size_t)row * p.H + nx.z) * kD + 16 * g));
      }
      // ---- epilogue: final rows, or the partial state for the far-tile kernel
      alive = __all_sync(kAll, alive && wait_ph(pv_done, (gt - 1) & 1, 296));
      tc_fence_after();
      float* red = sRed + 1024;
      red[g * 128 + rho] = l_run;
      named_sync(2 + qd, 128);
      const float l_tot = (red[rho] + red[128 + rho]) + (red[256 + rho] + red[384 + rho]);
      const bool store = alive && *s_abort == 0;
      const bool has_far = jlo > 0 || jhi < nkb;
      // O (divided by the row sum for final rows) goes through the idle Cw
      // buffer, so that the stores to global memory are whole rows: after the
      // quarter's barrier each warp writes 8 rows of its quarter.
      const uint32_t os = smem_u32(sm + SL::cw);
      {
        const float sc = has_far ? 1.f : (l_tot > 0.f ? 1.f / l_tot : 0.f);
        uint32_t r[16];
        tmem_ld16(tO + lane_off + 16 * g, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          sts128(os + kRowB * rho + 64 * g + 4 * e,
                 make_uint4(__float_as_uint(__uint_as_float(r[e]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 1]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 2]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 3]) * sc)));
      }
      if (has_far && g == 0 && store && i0 + rho < n)
        partial_ml(p)[((size_t)start + i0 + rho) * p.H + h] = make_float2(m_run, l_tot);
      named_sync(2 + qd, 128);  // the quarter's 32 rows are staged
      if (store) {
        if (has_far) {
          // un-normalised fp32 rows (256 bytes): lanes 0-15 one row, 16-31 the next
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 32 * qd + 8 * g + 2 * k + (lane >> 4);
            const uint4 v = lds128(os + kRowB * rr + 16 * (lane & 15));
            if (i0 + rr < n)
              *reinterpret_cast<uint4*>(partial_o(p) + ((size_t)start + i0 + rr) * p.H * kD + h * kD +
                                        4 * (lane & 15)) = v;
          }
        } else {
          // final rows in the I/O type (128 bytes): lanes 8 a .. 8 a + 7 one row
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int rr = 32 * qd + 8 * g + 4 * k + (lane >> 3);
            const uint32_t a = os + kRowB * rr + 32 * (lane & 7);
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
              *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (tok * p.H + h) * kD + 8 * (lane & 7)) = w;
            }
          }
        }
      }
      // the next item's Q (its rows were prefetched into L1 before the epilogue)
      if (nx.y >= 0) store_q(nx);
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
  cudaError_t e = cudaFuncSetAttribute(tc_near64_kernel<BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Smem::bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.max_items, near_sm_count());
  e = launch_after_plan(tc_near64_kernel<BF16>, grid, kThreads, Smem::bytes, s, p, maps);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_near64(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  return p.dtype == DF_BF16 ? launch_typed<true>(p, maps, s) : launch_typed<false>(p, maps, s);
}

}  // namespace dfa
