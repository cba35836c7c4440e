// Near-tile fused forward on tcgen05 (bf16 / fp16 I/O, fp32 accumulation), and
// the host orchestration of the tensor-core path (planning kernel -> near tiles
// -> far tiles).
//
// Operation: DisentangledFlash README "Status" (C2P/P2C disentangled attention,
// FP16/BF16, factorized padding masks, packed cu_seqlens) and the kernels-community
// "DisentangledFlash" discussion "Motivation" (exact, tiled and streaming, no
// [B,H,L,L] matrix).
//
// A near tile (128 queries x 128 keys whose relative distances are not all
// saturated) needs the band of PK / PQ rows [lo, lo + W), W <= 255, that its
// distances map to.  TMA stages Q, K, V and the band rows in 128-byte swizzled
// shared memory; tcgen05.mma forms S = Q.K^T, C = Q.PK[band]^T and
// P = K.PQ[band]^T (two 128-column halves) in tensor memory; the band products
// are drained to shared memory, rotated by 4 words per row so that both the
// drain and the gather are free of bank conflicts, and every score element
// gathers  C[i][idx(i-j) - lo] + P[j][idx(i-j) - lo].  The online softmax and
// P.V (P read back from tensor memory) follow.  Two warpgroups share every
// step of a tile: they split its key columns for the gather and the softmax
// (exchanging the row maximum through shared memory), warpgroup 0 drains the
// C band and warpgroup 1 the P band, and thread 0 issues the copies and MMAs.
// The next tile's K and band rows are fetched while the softmax runs, its V
// while the current P.V completes.
//
// A query block whose key range also has far tiles leaves its un-normalised
// partial state (O, running max, running sum) in the workspace for the
// far-tile kernel; otherwise this kernel writes the final rows.
#include "df_tc_common.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>

namespace dfa {

namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kTile = 128;

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
template <int D>
struct NearSmem {
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t q = 0;
  static constexpr uint32_t k = q + kChunks * kBoxBytes;
  static constexpr uint32_t v = k + kChunks * kBoxBytes;
  static constexpr uint32_t r = v + kChunks * kBoxBytes;  // PK band half, then drained C
  static constexpr uint32_t rp = r + 65536;               // PQ band half, then drained P
  // d = 64: the second band half (PK then PQ rows) lands with the first one
  static constexpr bool kBand1 = D == 64;
  static constexpr uint32_t br1 = rp + 65536;
  static constexpr uint32_t tab = br1 + (kBand1 ? 2 * kChunks * kBoxBytes : 0);  // int32 [256]
  static constexpr uint32_t colv = tab + 1024;            // float [128] key bias
  static constexpr uint32_t red = colv + 512;             // float [2][128]
  static constexpr uint32_t bars = red + 1024;
  static constexpr uint32_t tslot = bars + 64;
  static constexpr uint32_t bytes = tslot + 16;
  static constexpr uint32_t alloc = bytes;  // the base is 1024-byte aligned (checked)
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_near_kernel(const Problem p, const __grid_constant__ TcMaps maps) {
  using SL = NearSmem<D>;
  constexpr int kChunks = SL::kChunks;
  constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled tiles need 1024-byte aligned shared memory; the near-tile
  // layout uses the whole 227 KB, so there is no slack to realign at run time.
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(p.hdr, DF_ERR_CUDA, 250);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm + SL::q;
  uint8_t* sK = sm + SL::k;
  uint8_t* sV = sm + SL::v;
  uint8_t* sR = sm + SL::r;
  uint8_t* sRp = sm + SL::rp;
  uint8_t* sB1 = sm + SL::br1;
  int32_t* sTab = reinterpret_cast<int32_t*>(sm + SL::tab);
  float* sCol = reinterpret_cast<float*>(sm + SL::colv);
  float* sRed = reinterpret_cast<float*>(sm + SL::red);  // [2][128] cross-warpgroup exchange
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SL::bars);
  uint64_t* bar_q = bars;
  uint64_t* bar_kv = bars + 1;    // K and band half 0
  uint64_t* bar_v = bars + 2;
  uint64_t* bar_band = bars + 3;  // band half 1
  uint64_t* bar_mma = bars + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::tslot);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int half = warp >> 2;                   // warpgroup: key columns [64 half, 64 half + 64)
  const int row = (warp & 3) * 32 + (tid & 31);  // TMEM lane: query row (S, C, O) or key row (P)
  if (tid == 0) {
    for (int b = 0; b < 5; ++b) mbar_init(bars + b, 1);
    mbar_fence_init();
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
    tma_prefetch_desc(&maps.pk);
    tma_prefetch_desc(&maps.pq);
  }
  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  // S 0-127, C band 128-255, P band 256-383, O 384-(384 + D - 1)
  static_assert(tmem_region_fits(384, D, 512), "O accumulator in 512 columns");
  const uint32_t tS = tmem, tA = tmem + 128, tB = tmem + 256, tO = tmem + 384;

  uint32_t ph_q = 0, ph_kv = 0, ph_v = 0, ph_band = 0, ph_mma = 0;
  int failed_at = 0;
  const unsigned long long budget = p.wait_budget;
  // Block-uniform bounded wait.  On a timeout the phase is still awaited (with a
  // long fixed budget) so that no copy or MMA is in flight when the CTA leaves.
  auto wait_all = [&](uint64_t* bar, uint32_t& ph, int where) -> bool {
    const bool ok = mbar_wait(bar, ph, budget);
    const bool any_fail = __syncthreads_or(!ok) != 0;
    if (any_fail) {
      mbar_wait(bar, ph, kDrainBudget);
      if (failed_at == 0) failed_at = where;
    }
    ph ^= 1;
    return !any_fail;
  };

  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  const uint32_t sV_addr = smem_u32(sV);
  float* Cs = reinterpret_cast<float*>(sR);
  float* Ps = reinterpret_cast<float*>(sRp);

  // Work items are handed out dynamically, in list order (longest first): thread
  // 0 claims the next one from the counter in the workspace header (reset by
  // the planner) as the CTA finishes its previous item.
  volatile int* s_it = reinterpret_cast<volatile int*>(tslot + 1);
  for (;;) {
    if (tid == 0) *s_it = atomicAdd(&p.hdr->next_item, 1);
    __syncthreads();
    const int it = *s_it;
    __syncthreads();  // every thread has read it before thread 0 claims the next
    if (it >= n_items || failed_at != 0) break;
    const int4 item = p.items[it];
    const int start = item.x, n = item.y, h = item.z, i0 = item.w * kTile;
    const int nkb = (n + kTile - 1) / kTile;
    int jlo, jhi;
    near_block_range(i0, nkb, rsp, rsn, &jlo, &jhi);
    if (jhi <= jlo) continue;  // every tile is far: the far-tile kernel does the block
    const bool has_far = jlo > 0 || jhi < nkb;
    // K and band half 0 (and, with a dedicated buffer, half 1) of tile jb on one
    // barrier; lo and hi are idx at the tile's smallest and largest distance
    auto load_kband = [&](int jb, int lo, int hi) {
      const bool h1 = SL::kBand1 && hi - lo + 1 > 128;
      mbar_expect_tx(bar_kv, (h1 ? 5 : 3) * kChunks * kBoxBytes);
      for (int c = 0; c < kChunks; ++c) {
        tma_load_2d(sK + c * kBoxBytes, &maps.k, h * D + c * 64, start + jb * kTile, bar_kv);
        tma_load_2d(sR + c * kBoxBytes, &maps.pk, h * D + c * 64, lo, bar_kv);
        tma_load_2d(sRp + c * kBoxBytes, &maps.pq, h * D + c * 64, lo, bar_kv);
        if (h1) {
          tma_load_2d(sB1 + c * kBoxBytes, &maps.pk, h * D + c * 64, lo + 128, bar_kv);
          tma_load_2d(sB1 + (kChunks + c) * kBoxBytes, &maps.pq, h * D + c * 64, lo + 128, bar_kv);
        }
      }
    };
    auto idx_at = [&](int r) { return p.idx[r + p.lt - 1]; };
    auto load_v = [&](int jb) {
      mbar_expect_tx(bar_v, kChunks * kBoxBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(sV + c * kBoxBytes, &maps.v, h * D + c * 64, start + jb * kTile, bar_v);
    };
    if (tid == 0) {
      mbar_expect_tx(bar_q, kChunks * kBoxBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(sQ + c * kBoxBytes, &maps.q, h * D + c * 64, start + i0, bar_q);
      load_kband(jlo, idx_at(i0 - jlo * kTile - (kTile - 1)), idx_at(i0 - jlo * kTile + (kTile - 1)));
      load_v(jlo);
    }
    if (!wait_all(bar_q, ph_q, 1)) break;

    const int i = i0 + row;
    const size_t tok = (size_t)start + i;
    const bool row_in = i < n;
    float m_run = -INFINITY, l_run = 0.f;  // l_run: this warpgroup's columns only

    // raw index-table entries and the key bias of a tile, fetched one tile ahead
    auto fetch_tab = [&](int jb) -> int {
      return tid < 2 * kTile - 1 ? idx_at(i0 - jb * kTile - (kTile - 1) + tid) : 0;
    };
    auto fetch_col = [&](int jb) -> float {
      const int j = jb * kTile + tid;
      return tid < kTile ? (j < n ? p.keybias[(size_t)start + j] : -INFINITY) : 0.f;
    };
    int tab_next = fetch_tab(jlo);
    float col_next = fetch_col(jlo);
    for (int jb = jlo; jb < jhi; ++jb) {
      if (tid < 2 * kTile - 1) sTab[tid] = tab_next;
      if (tid < kTile) sCol[tid] = col_next;
      int lo_next = 0, hi_next = 0;
      if (jb + 1 < jhi) {
        tab_next = fetch_tab(jb + 1);
        col_next = fetch_col(jb + 1);
        if (tid == 0) {
          lo_next = tab_next;
          hi_next = idx_at(i0 - (jb + 1) * kTile + (kTile - 1));
        }
      }
      if (!wait_all(bar_kv, ph_kv, 2)) break;
      const int lo = sTab[0];
      const int W = sTab[2 * kTile - 2] - lo + 1;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tS, kmajor_desc(sQ, k), kmajor_desc(sK, k), kIdescQK, k > 0);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tA, kmajor_desc(sQ, k), kmajor_desc(sR, k), kIdescQK, k > 0);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tB, kmajor_desc(sK, k), kmajor_desc(sRp, k), kIdescQK, k > 0);
        mma_commit(bar_mma);
      }
      if (!wait_all(bar_mma, ph_mma, 3)) break;
      tc_fence_after();

      float x[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tS + lane_off + 64 * half, r0);
        tmem_ld32(tS + lane_off + 64 * half + 32, r1);
        tmem_ld_wait2(r0, r1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(r0[e]);
          x[32 + e] = __uint_as_float(r1[e]);
        }
      }

      const int nch = (W + 127) >> 7;
      bool ok = true;
      for (int hc = 0; hc < nch && ok; ++hc) {
        if (hc > 0) {
          const uint8_t* pk1 = SL::kBand1 ? sB1 : sR;
          const uint8_t* pq1 = SL::kBand1 ? sB1 + kChunks * kBoxBytes : sRp;
          if (!SL::kBand1) {
            if (tid == 0) {
              mbar_expect_tx(bar_band, 2 * kChunks * kBoxBytes);
              for (int c = 0; c < kChunks; ++c) {
                tma_load_2d(sR + c * kBoxBytes, &maps.pk, h * D + c * 64, lo + 128, bar_band);
                tma_load_2d(sRp + c * kBoxBytes, &maps.pq, h * D + c * 64, lo + 128, bar_band);
              }
            }
            if (!(ok = wait_all(bar_band, ph_band, 4))) break;
          }
          if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss(tA, kmajor_desc(sQ, k), kmajor_desc(pk1, k), kIdescQK, k > 0);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss(tB, kmajor_desc(sK, k), kmajor_desc(pq1, k), kIdescQK, k > 0);
            mma_commit(bar_mma);
          }
          if (!(ok = wait_all(bar_mma, ph_mma, 5))) break;
          tc_fence_after();
        }
        // drain: warpgroup 0 the C band (lane = query row), warpgroup 1 the P band
        // (lane = key row); every row is rotated by 4 * (row % 8) words
        {
          uint32_t r[32];
          const int rot = 4 * (row & 7);
          const uint32_t src = (half == 0 ? tA : tB) + lane_off;
          float* dst = (half == 0 ? Cs : Ps) + row * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(src + 32 * c, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int col = (32 * c + 4 * m + rot) & 127;
              *reinterpret_cast<uint4*>(dst + col) =
                  make_uint4(r[4 * m], r[4 * m + 1], r[4 * m + 2], r[4 * m + 3]);
            }
          }
        }
        tc_fence_before();
        __syncthreads();
        {
          const int base = lo + 128 * hc;  // the table holds raw idx values
          const float* crow = Cs + row * 128;
          const int crot = 4 * (row & 7);
          const int32_t* tab = sTab + row + kTile - 1 - 64 * half;
#pragma unroll
          for (int jj = 0; jj < 64; ++jj) {
            const int j = 64 * half + jj;
            const int u = tab[-jj] - base;
            if ((unsigned)u < 128u)
              x[jj] += crow[(u + crot) & 127] + Ps[j * 128 + ((u + 4 * (j & 7)) & 127)];
          }
        }
        fence_proxy_async_smem();
        __syncthreads();
      }
      if (!ok) break;
      // K and the band buffers are free: the next tile's K and band half 0 can land
      if (tid == 0 && jb + 1 < jhi) load_kband(jb + 1, lo_next, hi_next);

      // logits in log2 units; masked keys at -inf; row maximum over both warpgroups
      float mt = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < 64; jj += 4) {
        const float4 cv = *reinterpret_cast<const float4*>(sCol + 64 * half + jj);
        x[jj + 0] = fmaf(x[jj + 0], ks, cv.x);
        x[jj + 1] = fmaf(x[jj + 1], ks, cv.y);
        x[jj + 2] = fmaf(x[jj + 2], ks, cv.z);
        x[jj + 3] = fmaf(x[jj + 3], ks, cv.w);
        mt = fmaxf(mt, fmaxf(fmaxf(x[jj], x[jj + 1]), fmaxf(x[jj + 2], x[jj + 3])));
      }
      sRed[half * 128 + row] = mt;
      __syncthreads();
      mt = fmaxf(sRed[row], sRed[128 + row]);
      // Re-base only when the maximum grows by more than 2^8 (exact: numerator and
      // denominator share the stale base).  Both warpgroups take the same decision.
      float scale = 1.f;
      const bool rebase = mt > m_run + 8.f;
      if (rebase) {
        scale = ex2(m_run - mt);
        m_run = mt;
        l_run *= scale;
      }
      if (jb > jlo && __any_sync(0xffffffffu, rebase)) {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t a = tO + lane_off + half * (D / 2) + 32 * c;
          tmem_ld32(a, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
          tmem_st32(a, r);
        }
      }
      const float mb = m_run == -INFINITY ? 0.f : m_run;
      {
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = ex2(x[2 * e] - mb);
          const float p1 = ex2(x[2 * e + 1] - mb);
          l_run += p0 + p1;
          r[e] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
        }
        tmem_st32(tS + lane_off + 32 * half, r);
        tmem_st_wait();
      }
      if (!wait_all(bar_v, ph_v, 6)) break;  // includes the block barrier before P.V
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_ts(tO, tS + 8 * k, vtile_desc(sV_addr, k), kIdescPV, (jb > jlo || k > 0) ? 1u : 0u);
        mma_commit(bar_mma);
      }
      if (!wait_all(bar_mma, ph_mma, 7)) break;
      tc_fence_after();
      if (tid == 0 && jb + 1 < jhi) load_v(jb + 1);
    }
    if (failed_at) break;

    // epilogue: final rows, or the partial state for the far-tile kernel.  O
    // (divided by the row sum for final rows) goes through the idle band
    // buffer as fp32 rows of D words, 16-byte chunk c of row r at chunk
    // (c + r) mod (D / 4) (conflict-free both ways), so that the stores to
    // global memory are whole rows: warp w then writes rows 16 w .. 16 w + 15.
    sRed[half * 128 + row] = l_run;
    __syncthreads();
    const float l_tot = sRed[row] + sRed[128 + row];
    constexpr int kCpr = D / 4;  // 16-byte chunks per staged row
    const uint32_t os = smem_u32(Cs);
    {
      const float sc = has_far ? 1.f : (l_tot > 0.f ? 1.f / l_tot : 0.f);
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tmem_ld32(tO + lane_off + half * (D / 2) + 32 * c, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int ch = (half * (D / 2) + 32 * c + e) / 4;
          sts128(os + 16u * (uint32_t)(row * kCpr + (ch + row) % kCpr),
                 make_uint4(__float_as_uint(__uint_as_float(r[e]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 1]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 2]) * sc),
                            __float_as_uint(__uint_as_float(r[e + 3]) * sc)));
        }
      }
    }
    if (has_far && row_in && half == 0) partial_ml(p)[tok * p.H + h] = make_float2(m_run, l_tot);
    __syncthreads();  // every row is staged
    {
      const int lane = tid & 31;
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        const int rr = 16 * warp + k;  // staged row
        const int ir = i0 + rr;
        const size_t tr = (size_t)start + ir;
        if (has_far) {
          // fp32 row of D words: lanes take 16-byte chunks
          if (ir < n) {
#pragma unroll
            for (int c = lane; c < kCpr; c += 32) {
              const uint4 v = lds128(os + 16u * (uint32_t)(rr * kCpr + (c + rr) % kCpr));
              *reinterpret_cast<uint4*>(partial_o(p) + (tr * p.H + h) * D + 4 * c) = v;
            }
          }
        } else if (ir < n && p.keybias[tr] == 0.f) {
          // row of D values of the I/O type: lanes take 8 values (two chunks)
#pragma unroll
          for (int c = 2 * lane; c < kCpr; c += 64) {
            const uint4 v0 = lds128(os + 16u * (uint32_t)(rr * kCpr + (c + rr) % kCpr));
            const uint4 v1 = lds128(os + 16u * (uint32_t)(rr * kCpr + (c + 1 + rr) % kCpr));
            uint4 w;
            w.x = BF16 ? pack_bf16x2(__uint_as_float(v0.x), __uint_as_float(v0.y))
                       : pack_f16x2(__uint_as_float(v0.x), __uint_as_float(v0.y));
            w.y = BF16 ? pack_bf16x2(__uint_as_float(v0.z), __uint_as_float(v0.w))
                       : pack_f16x2(__uint_as_float(v0.z), __uint_as_float(v0.w));
            w.z = BF16 ? pack_bf16x2(__uint_as_float(v1.x), __uint_as_float(v1.y))
                       : pack_f16x2(__uint_as_float(v1.x), __uint_as_float(v1.y));
            w.w = BF16 ? pack_bf16x2(__uint_as_float(v1.z), __uint_as_float(v1.w))
                       : pack_f16x2(__uint_as_float(v1.z), __uint_as_float(v1.w));
            *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (tr * p.H + h) * D + 4 * c) = w;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (failed_at != 0 && tid == 0) raise_device_error(p.hdr, DF_ERR_DEVICE_TIMEOUT, 200 + failed_at);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

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

// Row-major [rows][row_elems] 16-bit matrix, 64 x 128 boxes, 128-byte swizzle.
// Row-major [rows][row_elems] 16-bit matrix in boxes of `inner` x 128 elements:
// 64-element boxes with the 128-byte swizzle, 16-element boxes with the 32-byte one.
bool encode_rows(CUtensorMap* m, const void* base, long long rows, long long row_elems, bool bf16,
                 int inner = 64) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
  const cuuint32_t box[2] = {(cuuint32_t)inner, 128};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
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
cudaError_t launch_near_typed(const Problem& p, const TcMaps& maps, cudaStream_t s) {
  const uint32_t bytes = NearSmem<D>::alloc;
  cudaError_t e = cudaFuncSetAttribute(tc_near_kernel<D, BF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.max_items, sm_count());
  tc_near_kernel<D, BF16><<<grid, kThreads, bytes, s>>>(p, maps);
  return cudaGetLastError();
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
  if (p.d == 64) {
    if (p.n_diag < 1 || !encode_rows(&maps.dpk, p.diag_pk, 256LL * p.n_diag, row, bf16) ||
        !encode_rows(&maps.dpq, p.diag_pq, 256LL * p.n_diag, row, bf16))
      return cudaErrorInvalidValue;
  } else {
    maps.dpk = maps.pk;
    maps.dpq = maps.pq;
  }
  if (ev0) cudaEventRecord(ev0, s);
  cudaError_t e;
  if (p.d == 64)
    e = launch_near64(p, maps, s);
  else
    e = bf16 ? launch_near_typed<128, true>(p, maps, s) : launch_near_typed<128, false>(p, maps, s);
  if (ev_mid) cudaEventRecord(ev_mid, s);
  // with no far tile possible the near-tile kernel writes every output row
  if (e == cudaSuccess && p.far_possible) e = launch_far(p, maps, s);
  if (ev1) cudaEventRecord(ev1, s);
  *launches = p.far_possible ? 2 : 1;
  return e;
}

}  // namespace dfa
