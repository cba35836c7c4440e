// Far-tile fused forward on tcgen05 (bf16 / fp16 I/O, fp32 accumulation).
//
// A far tile (128 queries x 128 keys) lies wholly in a saturated part of the
// DeBERTa relative-position index, so its c2p and p2c terms are the per-token
// scalars alpha_i = Q_i.PK[top or 0] and beta_j = K_j.PQ[top or 0]
// (DisentangledFlash README, "Status": C2P/P2C disentangled attention; the
// kernels-community "DisentangledFlash" discussion, "Motivation": exact,
// tiled, streaming).  What remains per tile is flash attention with a rank-1
// bias:  x_ij = (Q_i.K_j + beta_j) * log2(e)/sqrt(3d) + alpha_i.  beta_j enters
// the score MMA as a fifth K step: a selector block (1, 1, 0, 0, ...) or
// (0, 0, 1, 1, ...) for the tile's side times the keys' block of raw p2c terms
// (K.PQ[0] and K.PQ[top], each split into a 16-bit high and low part).
//
// Warp roles of one CTA (one CTA per SM, persistent over the work list):
//   warp 0      TMA producer of Q (two buffers, so the next item's Q lands
//               while the current one finishes), of K for every far tile and,
//               at d = 64, of V; K and V have separate stage barriers (a K
//               stage is free once its QK has completed, a V stage once its
//               P.V has);
//   warp 1      tcgen05.mma issuer of S = Q.K^T into a TMEM score buffer
//               (three at d = 64, P overwriting its S, so QK(G) waits only
//               for P(G - 3).V; at d = 128 this warp also issues the P.V);
//   warps 3, 2  at d = 64 the issuers of O_0 += P.V and O_1 += P.V for the
//               tiles of softmax warpgroup 0 and 1, with P read back from
//               TMEM: a P.V goes out as soon as its P is stored, never behind
//               the other warpgroup's blocking issue; at d = 128 warp 2 loads
//               V and warp 3 idles;
//   warps 4-7   softmax warpgroup 0: even far tiles, accumulator O_0;
//   warps 8-11  softmax warpgroup 1: odd far tiles, accumulator O_1.
// The control warpgroup gives registers back (setmaxnreg) so that each softmax
// thread can hold its 128-score row without spilling.
// The two warpgroups keep independent running (max, sum, O) so that neither
// waits for the other while the tensor core alternates between them; the two
// partial results are merged at the end of the item.  Warpgroup 0 starts from
// the partial state the near-tile kernel left for this query block.
#include "df_tc_common.cuh"

#include <algorithm>
#include <type_traits>

namespace dfa {

namespace {

using namespace ptx;

constexpr int kFarThreads = 384;
constexpr uint32_t kFarItemRing = 4;  // work items handed from warp 0 to the other roles

template <int D>
struct FarSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kStages = D == 64 ? 5 : 2;
  static constexpr uint32_t kTileBytes = kChunks * kBoxBytes;
  static constexpr uint32_t kStageBytes = 2 * kTileBytes + kAugBytes;
  static constexpr uint32_t q = 0;                                   // [2][Q tile]
  static constexpr uint32_t kv = q + 2 * kTileBytes;                 // [stage][K | V | key terms]
  static constexpr uint32_t sel = kv + kStages * kStageBytes;        // [2] selector blocks
  static constexpr uint32_t ml = sel + 2 * kAugBytes;                // float4 [2 wg][128]
  static constexpr uint32_t bars = ml + 2 * 128 * 16;
  // q_full[2], q_empty[2], k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[3],
  // p_full[2][2], o_final, drain[3], buf_free[3], sel_full
  static constexpr int kBars = 4 + 4 * kStages + 3 + 4 + 4 + 3 + 1 + 2 * kFarItemRing;
  static constexpr uint32_t misc = bars + kBars * 8;                 // abort flag, tmem slot,
                                                                     // softmax's current item
  static constexpr uint32_t ring = misc + 16;                        // int [kFarItemRing]
  static constexpr uint32_t bytes = ring + 4 * kFarItemRing;
  static constexpr uint32_t alloc = bytes + 1024;
};

struct ItemGeom {
  int start, n, h, i0, nkb, jlo, jhi, nt;
  __device__ __forceinline__ int block_of(int t) const { return t < jlo ? t : jhi + (t - jlo); }
  __device__ __forceinline__ bool pos_side(int t) const { return t < jlo; }
};

__device__ __forceinline__ ItemGeom item_geom(const Problem& p, int it, int rsp, int rsn) {
  const int4 item = p.items[it];
  ItemGeom g;
  g.start = item.x;
  g.n = item.y;
  g.h = item.z;
  g.i0 = item.w * 128;
  g.nkb = (g.n + 127) >> 7;
  near_block_range(g.i0, g.nkb, rsp, rsn, &g.jlo, &g.jhi);
  g.nt = g.jlo + (g.nkb - g.jhi);
  return g;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kFarThreads, 1)
    tc_far_kernel(const Problem p, const __grid_constant__ TcMaps maps) {
  using SL = FarSmem<D>;
  constexpr int kChunks = SL::kChunks;
  constexpr int S = SL::kStages;
  constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm + SL::q;
  uint8_t* sKV = sm + SL::kv;
  uint8_t* sSel = sm + SL::sel;
  float4* sML = reinterpret_cast<float4*>(sm + SL::ml);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SL::bars);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = bars + 4 + S;      // K(t) read: QK(t) has completed
  uint64_t* v_full = bars + 4 + 2 * S;
  uint64_t* v_empty = bars + 4 + 3 * S;  // V(t) read: P(t).V has completed
  uint64_t* s_full = bars + 4 + 4 * S;   // [3] S of the buffer computed
  // [wg][k & 1]: the four warps of warpgroup wg stored P of its k-th tile.  Two
  // per warpgroup because a warp may finish its next tile before a sibling
  // warp has stored the current one; it is never two tiles ahead, since its
  // next S waits for a P.V issued after this phase.
  uint64_t* p_full = s_full + 3;
  uint64_t* o_final = p_full + 4;
  uint64_t* drain = o_final + 1;         // [3]: one per MMA-issuing thread
  uint64_t* buf_free = drain + 3;  // [3] d = 64: the P.V that read the buffer is done
  uint64_t* sel_full = buf_free + 3;  // selector blocks landed
  // Work items: warp 0 claims the next item of the list (a global counter,
  // longest items first) when a ring slot is free and hands its index to the
  // other roles through the ring; a slot is free again once every consumer
  // (warp 1, warps 2 and 3 at d = 64 or warp 2 at d = 128, and the softmax
  // warpgroups' reader) has read it.  Index -1 ends the CTA's list.
  uint64_t* item_full = sel_full + 1;                // [kFarItemRing]
  uint64_t* item_empty = item_full + kFarItemRing;   // [kFarItemRing]
  volatile int* s_ring = reinterpret_cast<volatile int*>(sm + SL::ring);
  volatile int* s_cur = reinterpret_cast<volatile int*>(sm + SL::misc + 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SL::misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full + b, 1);
      mbar_init(q_empty + b, 1);
    }
    for (int s = 0; s < 4 * S; ++s) mbar_init(k_full + s, 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(buf_free + b, 1);
    }
    for (int b = 0; b < 4; ++b) mbar_init(p_full + b, 4);
    mbar_init(o_final, 1);  // d = 128: every P.V of the item done (d = 64 waits per tile)
    for (int b = 0; b < 3; ++b) mbar_init(drain + b, 1);
    mbar_init(sel_full, 1);
    for (uint32_t b = 0; b < kFarItemRing; ++b) {
      mbar_init(item_full + b, 1);
      mbar_init(item_empty + b, D == 64 ? 4 : 3);
    }
    *s_abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
    tma_prefetch_desc(&maps.kaug);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // TMEM columns of buffer b
  // d = 64: three score buffers (tile G of the CTA uses buffer G % 3) and the
  // two warpgroups' O; P(G) overwrites its own S once the softmax has read it,
  // so neither the softmax nor QK(G + 2) waits for a P.V.  d = 128: one score
  // buffer per warpgroup (P overwrites it) and the two O.
  constexpr bool kTriS = D == 64;
  constexpr uint32_t kScoreBufs = kTriS ? 3u : 2u, kOFirst = kTriS ? 384u : 256u;
  static_assert(tmem_region_fits(0, 128u * kScoreBufs, kOFirst), "score buffers below O");
  static_assert(tmem_region_fits(kOFirst, 2u * D, 512), "two O accumulators in 512 columns");
  const uint32_t tO_base = tmem + kOFirst;
  auto tS = [&](int b) { return tmem + 128u * b; };
  auto tO = [&](int b) { return tO_base + (uint32_t)D * b; };

  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const unsigned long long budget = p.wait_budget;
  df_ws_header* hdr = p.hdr;
  // warp 0: claim and hand out the c-th item; -1 at the end of the list (or
  // once the CTA aborts)
  auto claim_item = [&](uint32_t c) -> int {
    const uint32_t slot = c % kFarItemRing;
    if (c >= kFarItemRing &&
        !wait_or_abort(item_empty + slot, ((c / kFarItemRing) - 1) & 1, budget, s_abort, hdr, 330))
      return -1;
    if (*s_abort) return -1;
    int it = atomicAdd(&hdr->next_far_item, 1);
    if (it >= n_items) it = -1;
    s_ring[slot] = it;
    mbar_arrive(item_full + slot);  // release: the slot is visible to its waiters
    return it;
  };
  // any other role (one thread): the c-th item handed out
  auto take_item = [&](uint32_t c) -> int {
    const uint32_t slot = c % kFarItemRing;
    if (!wait_or_abort(item_full + slot, (c / kFarItemRing) & 1, budget, s_abort, hdr, 331)) return -1;
    const int it = s_ring[slot];
    mbar_arrive(item_empty + slot);
    return it;
  };

  if (warp == 0 || (!kTriS && warp == 2)) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: Q of every item and K of every far tile, and at d = 64 also V;
    // d = 128: warp 2 loads V.  K stages are released when QK has read them, V
    // stages when P.V has.
    setmaxnreg_dec<56>();
    if (lane == 0) {
      const bool is_k = warp == 0;
      const bool with_v = !is_k || kTriS;
      uint32_t g = 0, qc = 0, gk_issued = 0, gv_issued = 0, q_issued = 0;  // loads are issued in order
      if (is_k) {  // the two selector blocks, once
        mbar_expect_tx(sel_full, 2 * kAugBytes);
        tma_load_2d(sSel, &maps.kaug_sel, 0, 0, sel_full);
        tma_load_2d(sSel + kAugBytes, &maps.kaug_sel, 0, 128, sel_full);
      }
      for (uint32_t ci = 0;; ++ci) {
        const int it = is_k ? claim_item(ci) : take_item(ci);
        if (it < 0) break;
        const ItemGeom ig = item_geom(p, it, rsp, rsn);
        if (ig.nt == 0) continue;
        if (is_k) {
          const int qb = qc & 1;
          if (wait_or_abort(q_empty + qb, ((qc >> 1) & 1) ^ 1, budget, s_abort, hdr, 301)) {
            mbar_expect_tx(q_full + qb, SL::kTileBytes);
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d(sQ + qb * SL::kTileBytes + c * kBoxBytes, &maps.q, ig.h * D + c * 64,
                          ig.start + ig.i0, q_full + qb);
            q_issued = qc + 1;
          }
          ++qc;
        }
        for (int t = 0; t < ig.nt; ++t, ++g) {
          const int s = g % S;
          const int row = ig.start + ig.block_of(t) * 128;
          uint8_t* st = sKV + s * SL::kStageBytes;
          if (is_k && wait_or_abort(k_empty + s, ((g / S) & 1) ^ 1, budget, s_abort, hdr, 302)) {
            mbar_expect_tx(k_full + s, SL::kTileBytes + kAugBytes);
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d(st + c * kBoxBytes, &maps.k, ig.h * D + c * 64, row, k_full + s);
            // the keys' p2c terms, 16 values per key
            tma_load_2d(st + 2 * SL::kTileBytes, &maps.kaug, ig.h * 16, row, k_full + s);
            gk_issued = g + 1;
          }
          if (with_v && wait_or_abort(v_empty + s, ((g / S) & 1) ^ 1, budget, s_abort, hdr, 303)) {
            mbar_expect_tx(v_full + s, SL::kTileBytes);
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d(st + SL::kTileBytes + c * kBoxBytes, &maps.v, ig.h * D + c * 64, row, v_full + s);
            gv_issued = g + 1;
          }
        }
      }
      // no copy may still be landing when the CTA leaves: wait for the last load
      // issued into every stage and into both Q buffers
      for (uint32_t k = gk_issued > (uint32_t)S ? gk_issued - S : 0; k < gk_issued; ++k)
        mbar_wait(k_full + k % S, (k / S) & 1, kDrainBudget);
      for (uint32_t k = gv_issued > (uint32_t)S ? gv_issued - S : 0; k < gv_issued; ++k)
        mbar_wait(v_full + k % S, (k / S) & 1, kDrainBudget);
      for (uint32_t k = q_issued > 2 ? q_issued - 2 : 0; k < q_issued; ++k)
        mbar_wait(q_full + (k & 1), (k >> 1) & 1, kDrainBudget);
      if (is_k) mbar_wait(sel_full, 0, kDrainBudget);
    }
  } else if (warp == 1 || (kTriS && (warp == 2 || warp == 3))) {
    // ------------------------------------------------------------ MMA issuers
    // d = 64: warp 1 issues S = Q.K^T, warps 3 and 2 issue O_b += P.V for the
    // tiles of warpgroup 0 and 1, so that no chain waits behind another's
    // blocking issue (a P.V goes out as soon as its P is stored, not after the
    // other warpgroup's); every commit is made by the thread whose MMAs it
    // covers.  d = 128 (P overwrites S): warp 1 issues both in order.
    setmaxnreg_dec<56>();
    if (lane == 0) {
      const bool qk_role = warp == 1;
      const bool pv_role = warp != 1 || !kTriS;
      const int pv_wg = warp == 3 ? 0 : 1;  // d = 64: the warpgroup whose tiles this thread multiplies
      uint32_t g = 0, qc = 0;
      uint32_t pn[2] = {0, 0};  // tiles of warpgroup b whose P has been consumed
      const bool sel_ok = !qk_role || wait_or_abort(sel_full, 0, budget, s_abort, hdr, 316);
      const uint32_t kv_addr = smem_u32(sKV);
      for (uint32_t ci = 0;; ++ci) {
        const int it = take_item(ci);
        if (it < 0) break;
        const ItemGeom ig = item_geom(p, it, rsp, rsn);
        if (ig.nt == 0) continue;
        const bool has_partial = ig.jhi > ig.jlo;
        const int qb = qc & 1;
        const uint8_t* sQb = sQ + qb * SL::kTileBytes;
        const bool q_ok = qk_role && wait_or_abort(q_full + qb, (qc >> 1) & 1, budget, s_abort, hdr, 311);
        ++qc;
        auto issue_qk = [&](int t) {
          const uint32_t gs = g + t;
          const int s = gs % S;
          // score buffer: G % 3 at d = 64 (free once P(G - 3).V is done), else t % 2
          const int sb = kTriS ? (int)(gs % 3) : (t & 1);
          bool ok = true;
          if (kTriS && gs >= 3)
            ok = wait_or_abort(buf_free + sb, ((gs - 3) / 3) & 1, budget, s_abort, hdr, 314);
          ok = wait_or_abort(k_full + s, (gs / S) & 1, budget, s_abort, hdr, 312) && ok;
          if (ok && q_ok && sel_ok) {
            const uint64_t dq = kmajor_desc(sQb, 0);
            const uint64_t dk = kmajor_desc(sKV + s * SL::kStageBytes, 0);
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss(tS(sb), dq + kmajor_step(k), dk + kmajor_step(k), kIdescQK, k > 0);
            // S += selector . key terms: the p2c term of the tile's side (hi + lo)
            mma_ss(tS(sb), aug_desc(sSel + (ig.pos_side(t) ? kAugBytes : 0u)),
                   aug_desc(sKV + s * SL::kStageBytes + 2 * SL::kTileBytes), kIdescQK, 1u);
            mma_commit(s_full + sb);
            mma_commit(k_empty + s);
          }
        };
        auto issue_pv = [&](int t) {
          const int b = t & 1;
          const uint32_t gs = g + t;
          const int s = gs % S;
          const uint32_t k = pn[b]++;
          bool ok = wait_or_abort(p_full + 2 * b + (k & 1), (k >> 1) & 1, budget, s_abort, hdr, 313);
          ok = wait_or_abort(v_full + s, (gs / S) & 1, budget, s_abort, hdr, 315) && ok;
          if (ok) {
            const uint64_t dv = vtile_desc(kv_addr + s * SL::kStageBytes + SL::kTileBytes, 0);
            tc_fence_after();
            const bool carry = (t >= 2) || (b == 0 && has_partial);
            const uint32_t tP = tS(kTriS ? (int)(gs % 3) : b);  // P(t) overwrote its S
#pragma unroll
            for (int k = 0; k < 128 / 16; ++k)
              mma_ts(tO(b), tP + 8 * k, dv + vtile_step(k), kIdescPV, (k > 0 || carry) ? 1u : 0u);
            mma_commit(v_empty + s);
            if (kTriS) mma_commit(buf_free + (gs % 3));
          }
        };
        if (kTriS) {
          if (qk_role) {
            for (int t = 0; t < ig.nt; ++t) issue_qk(t);
          } else {
            for (int t = pv_wg; t < ig.nt; t += 2) issue_pv(t);
          }
        } else {
          // P overwrites S: QK(t) can only follow PV(t - 2)
          for (int t = 0; t <= ig.nt; ++t) {
            if (t < ig.nt) issue_qk(t);
            if (t >= 1) issue_pv(t - 1);
          }
        }
        g += ig.nt;
        if (qk_role) mma_commit(q_empty + qb);
        if (pv_role && !kTriS) mma_commit(o_final);
      }
      uint64_t* my_drain = drain + (warp == 1 ? 0 : warp == 3 ? 1 : 2);
      mma_commit(my_drain);
      mbar_wait(my_drain, 0, kDrainBudget);
    }
  } else if (warp == 3) {  // d = 128: idle (warp 2 loads V)
    setmaxnreg_dec<56>();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    setmaxnreg_inc<224>();
    const int wg = (warp - 4) >> 2;          // 0 or 1
    const int quad = warp & 3;               // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;        // query row inside the block
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float ks = p.kscale;
    // this warpgroup's O, in a register
    const uint32_t tOw = tO_base + (uint32_t)D * wg + lane_off;
    uint32_t sc = 0, ic = 0, own = 0, gbase = 0;  // gbase: CTA tiles before the item
    // Thread 0 of the warpgroups takes each item from the ring and leaves it in
    // s_cur; all 256 threads read it after their barrier, so that they run the
    // same list (a failed wait ends it for all of them).
    const bool reader = warp == 4 && lane == 0;
    uint32_t ci = 0;
    if (reader) *s_cur = take_item(ci++);
    named_sync(3, 256);
    for (;;) {
      const int it = *s_cur;
      if (it < 0) break;
      const ItemGeom ig = item_geom(p, it, rsp, rsn);
      if (ig.nt == 0) {  // (no item of the plan is empty) the item's end, without tiles
        named_sync(3, 256);  // every thread has read s_cur
        if (reader) *s_cur = take_item(ci++);
        named_sync(3, 256);
        continue;
      }
      const bool has_partial = ig.jhi > ig.jlo;
      const int i = ig.i0 + row;
      const bool row_in = i < ig.n;
      const size_t tok = (size_t)ig.start + i;
      const bool row_out = row_in && p.keybias[tok] == 0.f;
      const float* scal_h = p.scal + (size_t)ig.h * 4 * p.t_pad;
      const float a_neg = row_in ? scal_h[tok] : 0.f;
      const float a_pos = row_in ? scal_h[(size_t)p.t_pad + tok] : 0.f;
      float m_run = -INFINITY, l_run = 0.f;
      bool o_has = false;
      if (wg == 0 && has_partial) {
        // resume from the near-tile kernel's state of this query block
        uint32_t r[32];
        const float* src = partial_o(p) + (tok * p.H + ig.h) * D;
        if (row_in) {
          const float2 ml = partial_ml(p)[tok * p.H + ig.h];
          m_run = ml.x;
          l_run = ml.y;
        }
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 v = row_in ? *reinterpret_cast<const float4*>(src + 32 * c + e)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            r[e] = __float_as_uint(v.x);
            r[e + 1] = __float_as_uint(v.y);
            r[e + 2] = __float_as_uint(v.z);
            r[e + 3] = __float_as_uint(v.w);
          }
          tmem_st32(tO(0) + lane_off + 32 * c, r);
        }
        tmem_st_wait();
        o_has = true;
      }
      const float2 ks2 = make_float2(ks, ks);
      for (int t = wg; t < ig.nt; t += 2, ++own) {
        // score buffer of the tile: G % 3 (d = 64) or the warpgroup's own (d = 128)
        const uint32_t G = gbase + t;
        const int sb = kTriS ? (int)(G % 3) : wg;
        const uint32_t tSw = tmem + 128u * sb + lane_off;
        wait_or_abort(s_full + sb, kTriS ? (G / 3) & 1 : sc & 1, budget, s_abort, hdr, 321);
        ++sc;
        tc_fence_after();
        float x[128];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tSw, r0);
          tmem_ld32(tSw + 32, r1);
          tmem_ld32(tSw + 64, r2);
          tmem_ld32(tSw + 96, r3);
          tmem_ld_wait4(r0, r1, r2, r3);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(r0[e]);
            x[32 + e] = __uint_as_float(r1[e]);
            x[64 + e] = __uint_as_float(r2[e]);
            x[96 + e] = __uint_as_float(r3[e]);
          }
        }
        const float alpha = ig.pos_side(t) ? a_pos : a_neg;
        // Keys past the sequence end (only in its last key block) belong to the
        // next sequence or to nothing: their scores become -inf.
        const int kb = ig.block_of(t);
        if (kb == ig.nkb - 1 && (ig.n & 127) != 0) {
          const int valid = ig.n - 128 * kb;
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (j >= valid) x[j] = -INFINITY;
        }
        // row maximum of the raw scores (the key term came with S; the log2
        // scale is positive), eight independent chains
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
          const int a = (j >> 2) & 3;
          mx[2 * a] = fmax3(mx[2 * a], x[j], x[j + 1]);
          mx[2 * a + 1] = fmax3(mx[2 * a + 1], x[j + 2], x[j + 3]);
        }
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * ks + alpha;
        float scale = 1.f;
        const bool rebase = mt > m_run + 8.f;
        if (rebase) {
          scale = ex2(m_run - mt);
          m_run = mt;
          l_run *= scale;
        }
        // p = 2^(S ks + alpha - m), one FMA per pair; with no finite logit yet
        // every p is 0
        const float shift = m_run == -INFINITY ? INFINITY : m_run - alpha;
        const float2 nshift = make_float2(-shift, -shift);
        {
          uint32_t r[32];
          float2 acc[4];  // four independent sum chains
#pragma unroll
          for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float2 z = fma2(make_float2(x[64 * c + 2 * e], x[64 * c + 2 * e + 1]), ks2, nshift);
              const float2 pp = make_float2(ex2(z.x), ex2(z.y));
              acc[e & 3] = add2(acc[e & 3], pp);
              r[e] = BF16 ? pack_bf16x2(pp.x, pp.y) : pack_f16x2(pp.x, pp.y);
            }
            tmem_st32(tSw + 32 * c, r);  // P(t) overwrites the S it came from
          }
          const float2 s01 = add2(acc[0], acc[1]), s23 = add2(acc[2], acc[3]);
          l_run += (s01.x + s23.x) + (s01.y + s23.y);
        }
        // rescale O after the scores are dead (fewer live registers); P(t).V has
        // not been issued yet, so O still holds the tiles before t
        if (o_has && __any_sync(0xffffffffu, rebase)) {
          // d = 64: P(t - 2).V, this warpgroup's previous one, must be done (at
          // d = 128 the score MMA of t already followed it in the same pipe)
          if (kTriS && t >= 2) {
            wait_or_abort(buf_free + (G - 2) % 3, ((G - 2) / 3) & 1, budget, s_abort, hdr, 323);
            tc_fence_after();
          }
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(tOw + 32 * c, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
            tmem_st32(tOw + 32 * c, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 2 * wg + (own & 1));
        o_has = true;
      }
      // ---- merge the two warpgroups' partial results and write O
      if (kTriS) {
        // the last P.V into this warpgroup's O (its own issuer's, through the
        // tile's buffer); the other warpgroup waits for its own before the
        // barrier below, so both O are complete after it
        if (wg < ig.nt) {
          const uint32_t G = gbase + wg + 2 * ((ig.nt - 1 - wg) / 2);
          wait_or_abort(buf_free + G % 3, (G / 3) & 1, budget, s_abort, hdr, 322);
        }
      } else {
        wait_or_abort(o_final, ic & 1, budget, s_abort, hdr, 322);
        ++ic;
      }
      tc_fence_after();
      sML[wg * 128 + row] = make_float4(m_run, l_run, o_has ? 1.f : 0.f, 0.f);
      named_sync(3, 256);
      const float4 mine = sML[wg * 128 + row];
      const float4 other = sML[(1 - wg) * 128 + row];
      const float4 a = wg == 0 ? mine : other;   // warpgroup 0's state
      const float4 b = wg == 0 ? other : mine;   // warpgroup 1's state
      const bool ha = a.z != 0.f, hb = b.z != 0.f;
      float m = -INFINITY;
      if (ha) m = fmaxf(m, a.x);
      if (hb) m = fmaxf(m, b.x);
      const float fa = (ha && m != -INFINITY) ? ex2(a.x - m) : 0.f;
      const float fb = (hb && m != -INFINITY) ? ex2(b.x - m) : 0.f;
      const float l = a.y * fa + b.y * fb;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool store = row_out && *s_abort == 0;
      T* dst = static_cast<T*>(p.out) + (tok * p.H + ig.h) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = wg * (D / 2) + 32 * c;
        uint32_t ra[32], rb[32];
        tmem_ld32(tO(0) + lane_off + col, ra);
        tmem_ld32(tO(1) + lane_off + col, rb);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        if (store) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float o0 = (__uint_as_float(ra[2 * e]) * fa +
                              (hb ? __uint_as_float(rb[2 * e]) * fb : 0.f)) * inv;
            const float o1 = (__uint_as_float(ra[2 * e + 1]) * fa +
                              (hb ? __uint_as_float(rb[2 * e + 1]) * fb : 0.f)) * inv;
            w[e] = BF16 ? pack_bf16x2(o0, o1) : pack_f16x2(o0, o1);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      tc_fence_before();
      named_sync(3, 256);  // (also: every thread has read s_cur)
      gbase += ig.nt;
      if (reader) *s_cur = take_item(ci++);
      named_sync(3, 256);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

int far_sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

template <int D, bool BF16>
cudaError_t launch_far_typed(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  const uint32_t bytes = FarSmem<D>::alloc;
  cudaError_t e = cudaFuncSetAttribute(tc_far_kernel<D, BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the block's launched registers cover the split
  // (eight softmax warps at 224, four control warps at 56): refuse to launch if
  // the compiled register count does not
  static int regs_ok = -1;
  if (regs_ok < 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, tc_far_kernel<D, BF16>);
    if (e != cudaSuccess) return e;
    regs_ok = fa.numRegs * kFarThreads >= 256 * 224 + 128 * 56 ? 1 : 0;
  }
  if (!regs_ok) return cudaErrorInvalidConfiguration;
  const int grid = std::min(p.max_items, far_sm_count());
  tc_far_kernel<D, BF16><<<grid, kFarThreads, bytes, s>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_far(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  const bool bf16 = p.dtype == DF_BF16;
  if (p.d == 64) return bf16 ? launch_far_typed<64, true>(p, maps, s) : launch_far_typed<64, false>(p, maps, s);
  return bf16 ? launch_far_typed<128, true>(p, maps, s) : launch_far_typed<128, false>(p, maps, s);
}

}  // namespace dfa
