// Near-tile fused forward for head size 64 on tcgen05 (bf16 / fp16 I/O, fp32
// accumulation).
//
// Operation: DisentangledFlash README "Status" (C2P/P2C disentangled attention,
// FP16/BF16, packed cu_seqlens) and the kernels-community "DisentangledFlash"
// discussion "Motivation" (exact, tiled and streaming, no [B,H,L,L] matrix).
//
// Diagonal form of the position terms.  In a 128 x 128 tile with query block
// i0 and key block j0 = i0 - 128 m, element (i', j') has relative distance
// r = 128 m - 127 + t with t = i' - j' + 127, the tile's diagonal (0..254).
// The planning kernel stores, per offset m, the PK and PQ rows at idx(r) for
// every diagonal (the diagonal tables), so that two MMAs give
//     C[i'][t] = Q_i . PK[idx(r_t)]      P[j'][t] = K_j . PQ[idx(r_t)]
// and the score element needs C[i'][i' - j' + 127] + P[j'][i' - j' + 127]: a
// fixed skew, with no index lookups.  The 256 diagonal columns come in two MMA
// halves (t < 128, t >= 128) that share the tensor-memory columns A and B.
//
// Skew through shared memory.  Both terms are stored by query row, in the
// order the score row reads them:
//     Cw[i'][j'] = C[i'][i' - j' + 127]      Pw[i'][j'] = P[j'][i' - j' + 127]
// A lane of C drains its own query row, where consecutive diagonals are
// consecutive keys (descending): it converts two values per instruction and
// stores them as 32-bit words (rows of odd lanes start one key late, so their
// pairs are re-formed with a byte permute and the two end values go alone).  A
// lane of P (a key row) writes one 16-bit value into each query row.  The
// gather then reads 32 keys of each term as four 16-byte vectors and adds the
// two as fp16x2.  Rows are 272 bytes (16-byte aligned, 8 keys of padding): the
// vector loads are conflict free, the drains' stores at most 2-way.  The terms
// are rounded to fp16 (saturating) and scaled to log2 units when they are
// added; the upper triangle j' >= i' needs only the first half, so it is summed
// while the second half is in the tensor core.
//
// Roles (one CTA per SM, persistent over the work list):
//   warps 0-15  compute: warp w owns TMEM lanes 32 (w % 4) .. +31 (query rows
//               for S, C and O; key rows for P) and score columns
//               32 (w / 4) .. +31 of every tile; they drain, gather, run the
//               online softmax and write P (16-bit) into TMEM;
//   warp 16     control: TMA loads (Q; K, V double-buffered; the diagonal
//               table halves) and every tcgen05.mma, one elected thread.
// The MMAs of tile t + 1 (S, C and P first halves) are issued as soon as tile
// t has drained its second halves, so they run under tile t's gather and
// softmax.  Tensor memory: S 0-127, A 128-255, B 256-383, O 384-447,
// P 448-511.
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
constexpr int kThreads = kComputeThreads + 32;
constexpr uint32_t kRowB = 272;    // bytes per Cw / Pw row: 128 keys + 8 of padding
constexpr uint32_t kRowLead = 16;  // Cw lead: words written just before row 0 land here

struct Smem {
  static constexpr uint32_t q = 0;                       // Q tile
  static constexpr uint32_t k = q + kBoxBytes;           // K tiles [2]
  static constexpr uint32_t e0 = k + 2 * kBoxBytes;      // diagonal rows 0-127: PK | PQ
  static constexpr uint32_t e1 = e0 + 2 * kBoxBytes;     // diagonal rows 128-255: PK | PQ
  static constexpr uint32_t v = e1 + 2 * kBoxBytes;      // V tiles [2]
  static constexpr uint32_t cw = v + 2 * kBoxBytes;      // lead + fp16 [128][136]
  static constexpr uint32_t pw = cw + kRowLead + 128 * kRowB;  // fp16 [128][136]
  static constexpr uint32_t col = pw + 128 * kRowB;      // float [2][128] key bias
  static constexpr uint32_t red = col + 2 * 128 * 4;     // float [4][128]
  static constexpr uint32_t bars = red + 4 * 128 * 4;
  static constexpr int kBars = 15;
  static constexpr uint32_t misc = bars + kBars * 8;     // abort flag, TMEM slot
  static constexpr uint32_t bytes = misc + 16;
};
static_assert(Smem::bytes <= 227 * 1024, "near-tile shared memory");
static_assert(Smem::bars % 8 == 0, "mbarrier alignment");

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_near64_kernel(const Problem p, const __grid_constant__ TcMaps maps) {
  using SL = Smem;
  constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, kD, BF16 ? 1 : 0, 0, 1);
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(p.hdr, DF_ERR_CUDA, 260);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm + SL::q;
  uint8_t* sK = sm + SL::k;
  uint8_t* sE0 = sm + SL::e0;
  uint8_t* sE1 = sm + SL::e1;
  uint8_t* sV = sm + SL::v;
  float* sCol = reinterpret_cast<float*>(sm + SL::col);
  float* sRed = reinterpret_cast<float*>(sm + SL::red);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SL::bars);
  uint64_t* bar_q = bars + 0;
  uint64_t* bar_k = bars + 1;      // [2]
  uint64_t* bar_e0 = bars + 3;
  uint64_t* bar_e1 = bars + 4;
  uint64_t* bar_v = bars + 5;      // [2]
  uint64_t* bar_c1 = bars + 7;     // S, C and P first halves done
  uint64_t* bar_c2 = bars + 8;     // C and P second halves done
  uint64_t* bar_c3 = bars + 9;     // P.V done
  uint64_t* bar_d0 = bars + 10;    // first halves drained (one arrival per compute warp)
  uint64_t* bar_d1 = bars + 11;    // second halves drained
  uint64_t* bar_pr = bars + 12;    // P in TMEM
  uint64_t* bar_end = bars + 13;   // every MMA done (exit)
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SL::misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 10; ++b) mbar_init(bars + b, 1);
    mbar_init(bar_d0, kComputeWarps);
    mbar_init(bar_d1, kComputeWarps);
    mbar_init(bar_pr, kComputeWarps);
    mbar_init(bar_end, 1);
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
  const uint32_t tS = tmem, tA = tmem + 128, tB = tmem + 256, tO = tmem + 384, tP = tmem + 448;

  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const unsigned long long budget = p.wait_budget;
  df_ws_header* hdr = p.hdr;

  if (warp == kComputeWarps) {
    // ================================================================ control
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dpk);
      tma_prefetch_desc(&maps.dpq);
      // issued / consumed load counts per barrier (the n-th load on a barrier
      // completes its phase n & 1)
      uint32_t q_n = 0, k_n = 0, e0_n = 0, e1_n = 0, v_n = 0;
      uint32_t q_w = 0, k_w = 0, e0_w = 0, e1_w = 0, v_w = 0;
      uint32_t ph_c1 = 0, ph_c2 = 0, ph_c3 = 0, ph_d0 = 0, ph_d1 = 0, ph_pr = 0;
      // step-0 descriptors of the fixed buffers (K steps add kmajor_step)
      const uint64_t dq = kmajor_desc(sQ, 0);
      const uint64_t de0k = kmajor_desc(sE0, 0), de0q = kmajor_desc(sE0 + kBoxBytes, 0);
      const uint64_t de1k = kmajor_desc(sE1, 0), de1q = kmajor_desc(sE1 + kBoxBytes, 0);
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int4 item = p.items[it];
        const int start = item.x, n = item.y, h = item.z, ib = item.w;
        const int nkb = (n + kTile - 1) / kTile;
        int jlo, jhi;
        near_block_range(ib * kTile, nkb, rsp, rsn, &jlo, &jhi);
        const int nt = jhi - jlo;
        if (nt <= 0) continue;
        auto diag_row = [&](int t) {  // first row of tile t's block of the diagonal tables
          const int e = ib - (jlo + t) - p.diag_m0;
          if (e < 0 || e >= p.n_diag) {
            raise_device_error(hdr, DF_ERR_INVALID_ARG, 261);
            return 0;
          }
          return e * 256;
        };
        auto load_k = [&](int t) {  // K of tile t into buffer (k_n & 1)
          if (*s_abort) return;
          uint64_t* b = bar_k + (k_n & 1);
          mbar_expect_tx(b, kBoxBytes);
          tma_load_2d(sK + (k_n & 1) * kBoxBytes, &maps.k, h * kD, start + (jlo + t) * kTile, b);
          ++k_n;
        };
        auto load_v = [&](int t) {
          if (*s_abort) return;
          uint64_t* b = bar_v + (v_n & 1);
          mbar_expect_tx(b, kBoxBytes);
          tma_load_2d(sV + (v_n & 1) * kBoxBytes, &maps.v, h * kD, start + (jlo + t) * kTile, b);
          ++v_n;
        };
        auto load_e = [&](int t, int half) {
          if (*s_abort) return;
          uint64_t* b = half ? bar_e1 : bar_e0;
          uint8_t* dst = half ? sE1 : sE0;
          const int row = diag_row(t) + 128 * half;
          mbar_expect_tx(b, 2 * kBoxBytes);
          tma_load_2d(dst, &maps.dpk, h * kD, row, b);
          tma_load_2d(dst + kBoxBytes, &maps.dpq, h * kD, row, b);
          ++(half ? e1_n : e0_n);
        };
        auto wait_k = [&](int where) {  // the oldest load not yet consumed
          const bool ok = wait_or_abort(bar_k + (k_w & 1), (k_w >> 1) & 1, budget, s_abort, hdr, where);
          ++k_w;
          return ok;
        };
        auto wait_v = [&](int where) {
          const bool ok = wait_or_abort(bar_v + (v_w & 1), (v_w >> 1) & 1, budget, s_abort, hdr, where);
          ++v_w;
          return ok;
        };
        auto wait_e = [&](int half, int where) {
          uint32_t& w = half ? e1_w : e0_w;
          const bool ok = wait_or_abort(half ? bar_e1 : bar_e0, w & 1, budget, s_abort, hdr, where);
          ++w;
          return ok;
        };
        auto wait_ph = [&](uint64_t* bar, uint32_t& ph, int where) {
          const bool ok = wait_or_abort(bar, ph, budget, s_abort, hdr, where);
          ph ^= 1;
          return ok;
        };
        const uint32_t kbuf0 = k_n & 1;  // buffer of tile 0's K (tiles alternate)
        const uint32_t vbuf0 = v_n & 1;
        auto issue_mma1 = [&](int t) {
          const uint64_t dk = kmajor_desc(sK + ((kbuf0 + t) & 1) * kBoxBytes, 0);
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_ss(tS, dq + kmajor_step(k), dk + kmajor_step(k), kIdescQK, k > 0);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_ss(tA, dq + kmajor_step(k), de0k + kmajor_step(k), kIdescQK, k > 0);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_ss(tB, dk + kmajor_step(k), de0q + kmajor_step(k), kIdescQK, k > 0);
          mma_commit(bar_c1);
        };

        // ---- prologue: Q, K(0..1), diagonal halves of tile 0, V(0..1)
        mbar_expect_tx(bar_q, kBoxBytes);
        tma_load_2d(sQ, &maps.q, h * kD, start + ib * kTile, bar_q);
        ++q_n;
        load_k(0);
        if (nt > 1) load_k(1);
        load_e(0, 0);
        load_e(0, 1);
        load_v(0);
        if (nt > 1) load_v(1);
        bool ok = wait_or_abort(bar_q, q_w & 1, budget, s_abort, hdr, 270);
        ++q_w;
        ok = wait_k(271) && ok;
        ok = wait_e(0, 272) && ok;
        if (ok) issue_mma1(0);

        for (int t = 0; t < nt; ++t) {
          // (1) first halves done: diagonal half 0 is free for tile t + 1
          wait_ph(bar_c1, ph_c1, 273);
          if (t + 1 < nt) load_e(t + 1, 0);
          // (2) second halves, once the first ones are drained out of A and B
          ok = wait_ph(bar_d0, ph_d0, 274);
          ok = wait_e(1, 275) && ok;
          if (ok) {
            const uint64_t dk = kmajor_desc(sK + ((kbuf0 + t) & 1) * kBoxBytes, 0);
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_ss(tA, dq + kmajor_step(k), de1k + kmajor_step(k), kIdescQK, k > 0);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_ss(tB, dk + kmajor_step(k), de1q + kmajor_step(k), kIdescQK, k > 0);
            mma_commit(bar_c2);
          }
          // (3) K(t) and diagonal half 1 are free; tile t + 1's first MMAs go out
          //     when A and B are drained again
          wait_ph(bar_c2, ph_c2, 276);
          if (t + 1 < nt) load_e(t + 1, 1);
          if (t + 2 < nt) load_k(t + 2);
          ok = wait_ph(bar_d1, ph_d1, 277);
          if (t + 1 < nt) {
            ok = wait_k(278) && ok;
            ok = wait_e(0, 279) && ok;
            if (ok) issue_mma1(t + 1);
          }
          // (4) P(t).V
          ok = wait_ph(bar_pr, ph_pr, 280);
          ok = wait_v(281) && ok;
          if (ok) {
            const uint64_t dv = vtile_desc(smem_u32(sV + ((vbuf0 + t) & 1) * kBoxBytes), 0);
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)
              mma_ts(tO, tP + 8 * k, dv + vtile_step(k), kIdescPV, (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(bar_c3);
          }
          // (5) V(t)'s buffer takes V(t + 2) once P(t).V is done
          wait_ph(bar_c3, ph_c3, 282);
          if (t + 2 < nt) load_v(t + 2);
        }
      }
      // no copy or MMA may still be in flight when the CTA leaves
      for (; q_w < q_n; ++q_w) mbar_wait(bar_q, q_w & 1, kDrainBudget);
      for (; k_w < k_n; ++k_w) mbar_wait(bar_k + (k_w & 1), (k_w >> 1) & 1, kDrainBudget);
      for (; e0_w < e0_n; ++e0_w) mbar_wait(bar_e0, e0_w & 1, kDrainBudget);
      for (; e1_w < e1_n; ++e1_w) mbar_wait(bar_e1, e1_w & 1, kDrainBudget);
      for (; v_w < v_n; ++v_w) mbar_wait(bar_v + (v_w & 1), (v_w >> 1) & 1, kDrainBudget);
      mma_commit(bar_end);
      mbar_wait(bar_end, 0, kDrainBudget);
    }
  } else {
    // ================================================================ compute
    const int g = warp >> 2;             // score columns 32 g .. 32 g + 31
    const int qd = warp & 3;             // TMEM lane quarter
    const int rho = qd * 32 + lane;      // TMEM lane: query row (S, C, O) or key row (P)
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float ks = p.kscale;
    // 32-bit shared addresses of the fp16 rows (kRowB bytes each)
    const uint32_t cw = smem_u32(sm + SL::cw) + kRowLead, pw = smem_u32(sm + SL::pw);
    const uint32_t cw_row = cw + kRowB * rho;                       // C: lane rho's own row
    const uint32_t dP = pw + (uint32_t)((int)kRowB * (rho - 127) + 2 * rho);  // + kRowB t
    // gather of (rho, 32 g .. 32 g + 31): 64 bytes of each term's row
    const uint32_t gC = cw_row + 64u * g, gP = pw + kRowB * rho + 64u * g;

    uint32_t ph_c1 = 0, ph_c2 = 0, ph_c3 = 0, gt = 0;
    auto wait_ph = [&](uint64_t* bar, uint32_t& ph, int where) {
      const bool ok = wait_or_abort(bar, ph, budget, s_abort, hdr, where);
      ph ^= 1;
      return ok;
    };
    // Store NC drained columns t0 .. t0 + NC - 1 (t0 even) as fp16.  q[k] holds
    // columns t0 + 2k (bits 16-31) and t0 + 2k + 1 (bits 0-15).  EDGE chunks
    // reach outside the lane's window and test each store.
    auto store_c = [&](auto nc_tag, auto edge_tag, int t0, const uint32_t* q) {
      constexpr int NC = decltype(nc_tag)::value;
      constexpr bool EDGE = decltype(edge_tag)::value;
      // key u = rho + 127 - t of column t: the chunk covers keys a .. a + NC - 1,
      // column t0 + NC - 1 - (u - a) at key u.  Words at even keys; an odd row
      // (a odd) shifts every pair by one key.  A word written next to the row's
      // keys 0..127 lands in padding (keys -8..-1 and 128..135).
      const int a = rho + 128 - t0 - NC;
      const int odd = rho & 1;
      const uint32_t sel = odd ? 0x5432u : 0x3210u;
      const uint32_t base = cw_row + 2u * (uint32_t)(a + odd);
#pragma unroll
      for (int m = 0; m < NC / 2 - 1; ++m) {
        const uint32_t w = prmt(q[NC / 2 - 1 - m], q[NC / 2 - 2 - m], sel);
        if (!EDGE || (unsigned)(a + odd + 2 * m + 8) < 143u) sts32(base + 4u * m, w);
      }
      if (!odd) {
        if (!EDGE || (unsigned)(a + NC - 2 + 8) < 143u) sts32(base + 4u * (NC / 2 - 1), q[0]);
      } else {
        if (!EDGE || (unsigned)(a + 8) < 143u) sts16_lo(cw_row + 2u * (uint32_t)a, q[NC / 2 - 1]);
        if (!EDGE || (unsigned)(a + NC - 1 + 8) < 143u)
          sts16_lo(cw_row + 2u * (uint32_t)(a + NC - 1), q[0] >> 16);
      }
    };
    auto store_p = [&](auto nc_tag, auto edge_tag, int t0, const uint32_t* q) {
      constexpr int NC = decltype(nc_tag)::value;
      constexpr bool EDGE = decltype(edge_tag)::value;
      // column t of key row rho goes to query row t - 127 + rho
      const uint32_t dst = dP + kRowB * (uint32_t)t0;
#pragma unroll
      for (int k = 0; k < NC / 2; ++k) {
        if (!EDGE || (unsigned)(t0 + 2 * k - 127 + rho) < 128u) sts16_lo(dst + kRowB * (2 * k), q[k] >> 16);
        if (!EDGE || (unsigned)(t0 + 2 * k + 1 - 127 + rho) < 128u) sts16_lo(dst + kRowB * (2 * k + 1), q[k]);
      }
    };
    // Drain NC columns t0 .. t0 + NC - 1 (NC = 16 or 8) of A (side 0, C) or B
    // (side 1, P).
    auto drain = [&](auto nc_tag, int side, int t0, bool edge) {
      constexpr int NC = decltype(nc_tag)::value;
      uint32_t r[NC];
      const uint32_t src = (side ? tB : tA) + lane_off + (t0 & 127);
      if constexpr (NC == 16) {
        tmem_ld16(src, r);
      } else {
        tmem_ld8(src, r);
      }
      tmem_ld_wait(r);
      uint32_t q[NC / 2];
#pragma unroll
      for (int k = 0; k < NC / 2; ++k)
        q[k] = f16x2_satfinite(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
      using E1 = std::integral_constant<bool, true>;
      using E0 = std::integral_constant<bool, false>;
      if (side == 0) {
        if (edge) store_c(nc_tag, E1{}, t0, q); else store_c(nc_tag, E0{}, t0, q);
      } else {
        if (edge) store_p(nc_tag, E1{}, t0, q); else store_p(nc_tag, E0{}, t0, q);
      }
    };
    // The five 32-column chunks a lane quarter needs from one half:
    //   half 0: C chunks qd..3, P chunks 3-qd..3;  half 1: C chunks 0..qd, P chunks 0..3-qd
    //   (edge chunks: C chunk qd and P chunk 3 - qd of either half).
    // Warp g drains chunk g whole and 8 columns of the fifth one.
    auto drain_half = [&](int half) {
      auto chunk = [&](int item, int* side, int* c) {
        if (half == 0) {
          *side = item < 4 - qd ? 0 : 1;
          *c = *side == 0 ? qd + item : 3 - qd + (item - (4 - qd));
        } else {
          *side = item <= qd ? 0 : 1;
          *c = *side == 0 ? item : item - (qd + 1);
        }
      };
      int side, c;
      chunk(g, &side, &c);
      // the whole chunk in two 16-column loads (fewer live registers)
      drain(std::integral_constant<int, 16>{}, side, 128 * half + 32 * c,
            c == (side == 0 ? qd : 3 - qd));
      drain(std::integral_constant<int, 16>{}, side, 128 * half + 32 * c + 16,
            c == (side == 0 ? qd : 3 - qd));
      chunk(4, &side, &c);
      drain(std::integral_constant<int, 8>{}, side, 128 * half + 32 * c + 8 * g,
            c == (side == 0 ? qd : 3 - qd));
    };
    // Add the position terms of this thread's 32 elements.  Blocks wholly in the
    // upper triangle (j' >= rho: first halves only) are summed while the second
    // halves are in the tensor core; the rest, diagonal blocks included, after.
    auto gather = [&](float (&x)[32]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 c4 = lds128(gC + 16u * k), p4 = lds128(gP + 16u * k);
        const uint32_t cv[4] = {c4.x, c4.y, c4.z, c4.w}, pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 sum = f16x2_sum_f32x2(cv[w], pv[w]);
          x[8 * k + 2 * w] = fmaf(sum.x, ks, x[8 * k + 2 * w]);
          x[8 * k + 2 * w + 1] = fmaf(sum.y, ks, x[8 * k + 2 * w + 1]);
        }
      }
    };

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int4 item = p.items[it];
      const int start = item.x, n = item.y, h = item.z, i0 = item.w * kTile;
      const int nkb = (n + kTile - 1) / kTile;
      int jlo, jhi;
      near_block_range(i0, nkb, rsp, rsn, &jlo, &jhi);
      const int nt = jhi - jlo;
      if (nt <= 0) continue;
      const bool has_far = jlo > 0 || jhi < nkb;
      const int i = i0 + rho;
      const size_t tok = (size_t)start + i;
      const bool row_in = i < n;
      const bool row_out = row_in && p.keybias[tok] == 0.f;
      const int ctid = threadIdx.x;  // 0..511
      auto fetch_col = [&](int t) -> float {
        const int j = (jlo + t) * kTile + ctid;
        return ctid < kTile ? (j < n ? p.keybias[(size_t)start + j] : -INFINITY) : 0.f;
      };
      if (ctid < kTile) sCol[(gt & 1) * 128 + ctid] = fetch_col(0);
      float col_next = nt > 1 ? fetch_col(1) : 0.f;
      named_sync(1, kComputeThreads);
      float m_run = -INFINITY, l_run = 0.f;  // l_run: this warp's 32 columns only

      for (int t = 0; t < nt; ++t, ++gt) {
        // ---- S(t) and the first halves
        wait_ph(bar_c1, ph_c1, 290);
        tc_fence_after();
        float x[32];
        {
          uint32_t r[32];
          tmem_ld32(tS + lane_off + 32 * g, r);
          tmem_ld_wait(r);
          const float* cb = sCol + (gt & 1) * 128 + 32 * g;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 c4 = *reinterpret_cast<const float4*>(cb + e);
            x[e + 0] = fmaf(__uint_as_float(r[e + 0]), ks, c4.x);
            x[e + 1] = fmaf(__uint_as_float(r[e + 1]), ks, c4.y);
            x[e + 2] = fmaf(__uint_as_float(r[e + 2]), ks, c4.z);
            x[e + 3] = fmaf(__uint_as_float(r[e + 3]), ks, c4.w);
          }
        }
        drain_half(0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_d0);
        named_sync(1, kComputeThreads);
        if (g > qd) gather(x);
        // ---- second halves
        wait_ph(bar_c2, ph_c2, 291);
        tc_fence_after();
        drain_half(1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_d1);
        named_sync(1, kComputeThreads);
        if (g <= qd) gather(x);

        // ---- online softmax (log2 units); row maximum over the four column groups
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, x[e]);
        sRed[g * 128 + rho] = mt;
        if (ctid < kTile && t + 1 < nt) sCol[((gt + 1) & 1) * 128 + ctid] = col_next;
        named_sync(1, kComputeThreads);
        if (t + 2 < nt) col_next = fetch_col(t + 2);
        mt = fmaxf(fmaxf(sRed[rho], sRed[128 + rho]), fmaxf(sRed[256 + rho], sRed[384 + rho]));
        // Re-base only when the maximum grows by more than 2^8 (exact: numerator and
        // denominator share the stale base).  All four warps of a row agree.
        float scale = 1.f;
        const bool rebase = mt > m_run + 8.f;
        if (rebase) {
          scale = ex2(m_run - mt);
          m_run = mt;
          l_run *= scale;
        }
        // P(t - 1).V must be done before O is rescaled or P is overwritten
        if (t > 0) wait_ph(bar_c3, ph_c3, 292);
        tc_fence_after();
        if (t > 0 && __any_sync(0xffffffffu, rebase)) {
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
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(x[2 * e] - mb);
            const float p1 = ex2(x[2 * e + 1] - mb);
            acc = add2(acc, make_float2(p0, p1));
            r[e] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
          }
          l_run += acc.x + acc.y;
          tmem_st16(tP + lane_off + 16 * g, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pr);
      }

      // ---- epilogue: final rows, or the partial state for the far-tile kernel
      wait_ph(bar_c3, ph_c3, 293);
      tc_fence_after();
      sRed[g * 128 + rho] = l_run;
      named_sync(1, kComputeThreads);
      const float l_tot = (sRed[rho] + sRed[128 + rho]) + (sRed[256 + rho] + sRed[384 + rho]);
      uint32_t r[16];
      tmem_ld16(tO + lane_off + 16 * g, r);
      tmem_ld_wait(r);
      const bool store = *s_abort == 0;
      if (has_far) {
        if (row_in && store) {
          float* dst = partial_o(p) + (tok * p.H + h) * kD + 16 * g;
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<uint4*>(dst + e) = make_uint4(r[e], r[e + 1], r[e + 2], r[e + 3]);
          if (g == 0) partial_ml(p)[tok * p.H + h] = make_float2(m_run, l_tot);
        }
      } else if (row_out && store) {
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float o0 = __uint_as_float(r[2 * e]) * inv;
          const float o1 = __uint_as_float(r[2 * e + 1]) * inv;
          w[e] = BF16 ? pack_bf16x2(o0, o1) : pack_f16x2(o0, o1);
        }
        uint4* d4 = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (tok * p.H + h) * kD + 16 * g);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      // sRed is rewritten by the next item only after its first barriers
      named_sync(1, kComputeThreads);
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
  tc_near64_kernel<BF16><<<grid, kThreads, Smem::bytes, s>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_near64(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  return p.dtype == DF_BF16 ? launch_typed<true>(p, maps, s) : launch_typed<false>(p, maps, s);
}

}  // namespace dfa
