// Backward pass of the disentangled attention on CUDA cores (strict fp32).
//
// The pages stop at the forward (DisentangledFlash 0.2.0 README, "Status":
// training still takes the stock DeBERTa path); this file differentiates the
// same score
//   z_ij = (Q_i.K_j + Q_i.PK[idx(i-j)] + K_j.PQ[idx(i-j)]) / sqrt(3 d)
// with the tiled, streaming evaluation of the kernels-community
// "DisentangledFlash" discussion ("Motivation"): no n x n matrix leaves shared
// memory.  With p the softmax, dP_ij = dO_i.V_j, D_i = dO_i.O_i and
// dS_ij = p_ij (dP_ij - D_i) / sqrt(3 d):
//   dV_j = sum_i p_ij dO_i         dQ_i = sum_j dS_ij (K_j + PK[idx_ij])
//   dK_j = sum_i dS_ij (Q_i + PQ[idx_ij])
//   dPK[r] = sum_{idx_ij = r} dS_ij Q_i,   dPQ[r] = sum_{idx_ij = r} dS_ij K_j
//
// Launches (one stream, in order):
//   query kernel  per 64 query rows: pass 1 is the forward in fp32 (row
//                 log-sum-exp and O, hence D_i); pass 2 recomputes the tiles,
//                 forms dS, accumulates dQ = dS.K and the bucket sums
//                 G_c2p[i][r] = sum_{j: idx_ij = r} dS_ij.
//   key kernel    per 64 keys: recomputes the tiles with the stored row
//                 statistics, accumulates dV = P^T.dO, dK = dS^T.Q and the
//                 bucket sums G_p2c[j][r].
// The bucket sums go to the zero-initialised global tables with atomic adds
// from near tiles; a far tile has a single relative index, so its row (column)
// sums stay in registers for the whole block and are added once at the end.
//   GEMMs         dQ += G_c2p.PK, dK += G_p2c.PQ, and dPK = G_c2p^T.Q,
//                 dPQ = G_p2c^T.K reduced over fixed token ranges (partial
//                 sums, then one summing kernel; no global atomics).
// Score tiles are 64 x 64 with 4 x 4 register micro-tiles (rows ty + 16 a,
// columns tx + 16 b) as in the strict-fp32 forward; the position terms of a
// near tile come from the PK / PQ rows of the tile's index band, and a far
// tile (every distance saturated) uses the per-token scalars of the planner.
#include "df_common.cuh"

#include <math.h>

#include <algorithm>

namespace dfa {

namespace {

constexpr int BM = 64;   // query rows per tile
constexpr int BN = 64;   // keys per tile
constexpr int DC = 32;   // head-dim chunk staged at once
constexpr int WB = 128;  // index-band capacity (BM + BN - 1 rows)
constexpr int kThreads = 256;
static_assert(BM == BN, "query and key chunks are staged by one loop");

// Shared-memory map of the two tile kernels, in floats.
struct BwdSmem {
  static constexpr int q = 0;                      // [DC][BM + 1] query chunk
  static constexpr int k = q + DC * (BM + 1);      // [DC][BN + 1] key chunk
  static constexpr int g = k + DC * (BN + 1);      // [DC][BM + 1] dO chunk
  static constexpr int v = g + DC * (BM + 1);      // [DC][BN + 1] V chunk
  static constexpr int pk = v + DC * (BN + 1);     // [DC][WB + 1] PK band; later tile A [BM][BN]
  static constexpr int pq = pk + DC * (WB + 1);    // [DC][WB + 1] PQ band; later tile B [BM][BN]
  static constexpr int rowA = pq + DC * (WB + 1);  // [2][BM] query scalars (neg, pos side)
  static constexpr int colB = rowA + 2 * BM;       // [3][BN] key scalars (neg, pos), key bias
  static constexpr int floats = colB + 3 * BN;
  static_assert(BM * BN <= DC * (WB + 1), "tiles A and B reuse the band buffers");
  // pass 1 of the query kernel keeps V [BN][D] and P [BM][BN + 1] in the dO,
  // V and band buffers, which it does not otherwise use after the scores
  static constexpr int pass1 = g;
  static constexpr int pass1_floats = pk + 2 * DC * (WB + 1) - g;
  static_assert(BN * 128 + BM * (BN + 1) <= pass1_floats, "pass-1 V and P fit at d = 128");
};

struct TileGeom {
  bool far_pos, far_neg, far;
  int lo, w;
  int col[7];  // band row of diagonal ty - tx + 16 (dd - 3), relative to lo
};

__device__ __forceinline__ void tile_geom(const Problem& p, int rsp, int rsn, int i0, int j0, int ty,
                                          int tx, TileGeom& g) {
  const int rlo = i0 - j0 - (BN - 1), rhi = i0 - j0 + (BM - 1);
  g.far_pos = rlo >= rsp;
  g.far_neg = rhi <= rsn;
  g.far = g.far_pos || g.far_neg;
  g.lo = 0;
  g.w = 0;
#pragma unroll
  for (int dd = 0; dd < 7; ++dd) g.col[dd] = 0;
  if (!g.far) {
    g.lo = p.idx[rlo + p.lt - 1];
    g.w = p.idx[rhi + p.lt - 1] - g.lo + 1;
#pragma unroll
    for (int dd = 0; dd < 7; ++dd) g.col[dd] = p.idx[i0 - j0 + ty - tx + 16 * (dd - 3) + p.lt - 1] - g.lo;
  }
}

// dst[c * STRIDE + r] = fp32 of row r, column c (c < DC) of a [rows][ts]
// array starting at `base`, for r < rows; rows at or past `lim` read as 0.
// Each thread moves 16-byte vectors; within a warp the transposed stores hit
// 32 different banks (STRIDE = 1 modulo 32).
template <typename T, int STRIDE>
__device__ __forceinline__ void stage_t(const T* __restrict__ base, size_t ts, int rows, int lim,
                                        float* dst) {
  constexpr int V = 16 / sizeof(T);  // elements per vector
  constexpr int VPR = DC / V;        // vectors per row
  static_assert(STRIDE % 32 == 1, "conflict-free transposed stores");
  for (int e = threadIdx.x; e < rows * VPR; e += kThreads) {
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

// Raw score of tile (i0, j0): s = Q.K^T, plus for a near tile the position
// products Q_i.PK[idx] + K_j.PQ[idx] in the same accumulator; with DP also
// dp = dO.V^T.  Also stages the query / key scalars of the tile.  Every kernel
// forms the scores through this function, so they agree to the last bit.
template <typename T, int D, bool DP>
__device__ __forceinline__ void score_tile(const Problem& p, const T* __restrict__ gdo,
                                           const float* scal_h, int start, int n, int h, int i0,
                                           int j0, const TileGeom& g, float* sm, float (&s)[4][4],
                                           float (&dp)[4][4]) {
  const T* __restrict__ gq = static_cast<const T*>(p.q);
  const T* __restrict__ gk = static_cast<const T*>(p.k);
  const T* __restrict__ gv = static_cast<const T*>(p.v);
  const T* __restrict__ gpk = static_cast<const T*>(p.pk);
  const T* __restrict__ gpq = static_cast<const T*>(p.pq);
  float* Qs = sm + BwdSmem::q;
  float* Ks = sm + BwdSmem::k;
  float* Gs = sm + BwdSmem::g;
  float* Vc = sm + BwdSmem::v;
  float* PKs = sm + BwdSmem::pk;
  float* PQs = sm + BwdSmem::pq;
  float* rowA = sm + BwdSmem::rowA;
  float* colB = sm + BwdSmem::colB;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const size_t ts = (size_t)p.H * D;
  __syncthreads();  // every reader of the staging buffers and scalars is done
  for (int e = tid; e < BM; e += kThreads) {
    const int t = start + i0 + e;
    rowA[e] = i0 + e < n ? scal_h[0 * (size_t)p.t_pad + t] : 0.f;
    rowA[BM + e] = i0 + e < n ? scal_h[1 * (size_t)p.t_pad + t] : 0.f;
  }
  for (int e = tid; e < BN; e += kThreads) {
    const int t = start + j0 + e;
    const bool ok = j0 + e < n;
    colB[e] = ok ? scal_h[2 * (size_t)p.t_pad + t] : -INFINITY;
    colB[BN + e] = ok ? scal_h[3 * (size_t)p.t_pad + t] : -INFINITY;
    colB[2 * BN + e] = ok ? p.keybias[t] : -INFINITY;
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) s[a][b] = dp[a][b] = 0.f;
  for (int kc = 0; kc < D; kc += DC) {
    if (kc) __syncthreads();
    const size_t qrow = (size_t)(start + i0) * ts + (size_t)h * D + kc;
    const size_t krow = (size_t)(start + j0) * ts + (size_t)h * D + kc;
    stage_t<T, BM + 1>(gq + qrow, ts, BM, n - i0, Qs);
    stage_t<T, BN + 1>(gk + krow, ts, BN, n - j0, Ks);
    if (DP) {
      stage_t<T, BM + 1>(gdo + qrow, ts, BM, n - i0, Gs);
      stage_t<T, BN + 1>(gv + krow, ts, BN, n - j0, Vc);
    }
    if (!g.far) {
      const size_t prow = (size_t)g.lo * ts + (size_t)h * D + kc;
      stage_t<T, WB + 1>(gpk + prow, ts, g.w, g.w, PKs);
      stage_t<T, WB + 1>(gpq + prow, ts, g.w, g.w, PQs);
    }
    __syncthreads();
#pragma unroll 2
    for (int c = 0; c < DC; ++c) {
      float qa[4], kb[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qa[a] = Qs[c * (BM + 1) + ty + 16 * a];
#pragma unroll
      for (int b = 0; b < 4; ++b) kb[b] = Ks[c * (BN + 1) + tx + 16 * b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) s[a][b] = fmaf(qa[a], kb[b], s[a][b]);
      if (!g.far) {
        float pkd[7], pqd[7];
#pragma unroll
        for (int dd = 0; dd < 7; ++dd) {
          pkd[dd] = PKs[c * (WB + 1) + g.col[dd]];
          pqd[dd] = PQs[c * (WB + 1) + g.col[dd]];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            s[a][b] = fmaf(qa[a], pkd[a - b + 3], s[a][b]);
            s[a][b] = fmaf(kb[b], pqd[a - b + 3], s[a][b]);
          }
      }
      if (DP) {
        float ga[4], vb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) ga[a] = Gs[c * (BM + 1) + ty + 16 * a];
#pragma unroll
        for (int b = 0; b < 4; ++b) vb[b] = Vc[c * (BN + 1) + tx + 16 * b];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) dp[a][b] = fmaf(ga[a], vb[b], dp[a][b]);
      }
    }
  }
}

// Logits of the tile in log2 units (the forward's), -inf at masked and
// out-of-range keys.
__device__ __forceinline__ void tile_logits(const float* sm, const TileGeom& g, int n, int j0, float ks,
                                            const float (&s)[4][4], float (&x)[4][4]) {
  const float* rowA = sm + BwdSmem::rowA;
  const float* colB = sm + BwdSmem::colB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int jj = tx + 16 * b;
      float v;
      if (g.far) {
        const float al = g.far_pos ? rowA[BM + ty + 16 * a] : rowA[ty + 16 * a];
        const float be = g.far_pos ? colB[BN + jj] : colB[jj];
        v = fmaf(s[a][b], ks, al + be);
      } else {
        v = fmaf(s[a][b], ks, colB[2 * BN + jj]);
      }
      x[a][b] = j0 + jj < n ? v : -INFINITY;
    }
}

// Adds the tile's dS to the bucket sums.  G points at the table row of the
// block's first query row (BY_ROW) or key, rows H * R floats apart; `lim` is
// the number of rows inside the sequence.  Near tiles add each nonzero entry
// to the global table; a far tile has one relative index (bucket 0 or
// 2 span - 1), so its entries go to the per-thread sums `far` ([row or
// column u][side]), flushed by the caller.
template <bool BY_ROW>
__device__ __forceinline__ void bucket_sums(float* G, size_t row_stride, int lim, const TileGeom& g,
                                            const float (&ds)[4][4], float (&far)[4][2]) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  if (g.far) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += BY_ROW ? ds[u][e] : ds[e][u];
      if (g.far_pos)
        far[u][1] += sum;
      else
        far[u][0] += sum;
    }
  } else {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int row = BY_ROW ? ty + 16 * a : tx + 16 * b;
        if (row < lim && ds[a][b] != 0.f)
          atomicAdd(G + (size_t)row * row_stride + g.lo + g.col[a - b + 3], ds[a][b]);
      }
  }
}

// ---------------------------------------------------------------- query side
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 2 : 1) bwd_q_kernel(const BwdProblem b) {
  extern __shared__ float sm[];
  const Problem& p = b.f;
  constexpr int NC = D / 16;  // output columns per thread
  const T* __restrict__ gk = static_cast<const T*>(p.k);
  const T* __restrict__ gv = static_cast<const T*>(p.v);
  const T* __restrict__ gdo = static_cast<const T*>(b.dout);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H, R = b.R;
  const size_t ts = (size_t)H * D;
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  float* Vs = sm + BwdSmem::pass1;  // pass 1: [BN][D]
  float* Ps = Vs + BN * D;          // pass 1: [BM][BN + 1]
  float* tA = sm + BwdSmem::pk;     // pass 2: dS tile [BM][BN]
  float* Ks = sm + BwdSmem::k;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 item = p.items[it];
    const int start = item.x, n = item.y, h = item.z, qb = item.w;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    const int nkb = (n + BN - 1) / BN;
    for (int sub = 0; sub < kQBlock / BM; ++sub) {
      const int i0 = qb * kQBlock + sub * BM;
      if (i0 >= n) break;
      // ---- pass 1: the forward of these rows in fp32
      float m[4], l[4], o[4][NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) o[a][c] = 0.f;
      }
      for (int jb = 0; jb < nkb; ++jb) {
        const int j0 = jb * BN;
        TileGeom g;
        tile_geom(p, rsp, rsn, i0, j0, ty, tx, g);
        float s[4][4], dp[4][4], x[4][4];
        score_tile<T, D, false>(p, gdo, scal_h, start, n, h, i0, j0, g, sm, s, dp);
        tile_logits(sm, g, n, j0, ks, s, x);
        __syncthreads();  // V and P overwrite the band buffers
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float mt = fmaxf(fmaxf(x[a][0], x[a][1]), fmaxf(x[a][2], x[a][3]));
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
          const float mn = fmaxf(m[a], mt);
          const float base = mn == -INFINITY ? 0.f : mn;
          const float corr = exp2f(m[a] - base);
          m[a] = mn;
          l[a] *= corr;
#pragma unroll
          for (int c = 0; c < NC; ++c) o[a][c] *= corr;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const float pv = exp2f(x[a][bb] - base);
            l[a] += pv;
            Ps[(ty + 16 * a) * (BN + 1) + tx + 16 * bb] = pv;
          }
        }
        {
          constexpr int V = 16 / sizeof(T), VPR = D / V;
          for (int e = tid; e < BN * VPR; e += kThreads) {
            const int j = e / VPR, v = e % VPR;
            float4 f[V / 4];
            if (j0 + j < n) {
              const uint4 raw = *reinterpret_cast<const uint4*>(gv + (size_t)(start + j0 + j) * ts +
                                                                (size_t)h * D + v * V);
              const T* el = reinterpret_cast<const T*>(&raw);
#pragma unroll
              for (int k = 0; k < V / 4; ++k)
                f[k] = make_float4(IO<T>::to_f(el[4 * k]), IO<T>::to_f(el[4 * k + 1]),
                                   IO<T>::to_f(el[4 * k + 2]), IO<T>::to_f(el[4 * k + 3]));
            } else {
#pragma unroll
              for (int k = 0; k < V / 4; ++k) f[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < V / 4; ++k) reinterpret_cast<float4*>(Vs + j * D + v * V)[k] = f[k];
          }
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < BN; ++j) {
          float pa[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) pa[a] = Ps[(ty + 16 * a) * (BN + 1) + j];
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const float vv = Vs[j * D + tx + 16 * c];
#pragma unroll
            for (int a = 0; a < 4; ++a) o[a][c] = fmaf(pa[a], vv, o[a][c]);
          }
        }
      }
      // row statistics: log-sum-exp (log2 units) and D_i = dO_i . O_i; a
      // masked row has no output, so +inf makes every p of it 0
      float rL[4], rD[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float lt = l[a];
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        const int i = i0 + ty + 16 * a;
        const size_t t = (size_t)start + i;
        const bool in = i < n;
        const bool live = in && p.keybias[t] == 0.f;
        const float inv = 1.f / lt;
        float dsum = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          dsum = fmaf(in ? IO<T>::load(gdo + t * ts + (size_t)h * D + tx + 16 * c) : 0.f, o[a][c] * inv, dsum);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
        rL[a] = live ? m[a] + log2f(lt) : INFINITY;
        rD[a] = live ? dsum : 0.f;
        if (tx == 0 && in) {
          b.lse[t * H + h] = rL[a];
          b.drow[t * H + h] = rD[a];
        }
      }
      // ---- pass 2: dS, dQ = dS.K and the rows' bucket sums
      float* G = b.gc + ((size_t)(start + i0) * H + h) * R;
      float dq[4][NC], far[4][2];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        far[a][0] = far[a][1] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) dq[a][c] = 0.f;
      }
      for (int jb = 0; jb < nkb; ++jb) {
        const int j0 = jb * BN;
        TileGeom g;
        tile_geom(p, rsp, rsn, i0, j0, ty, tx, g);
        float s[4][4], dp[4][4], x[4][4], ds[4][4];
        score_tile<T, D, true>(p, gdo, scal_h, start, n, h, i0, j0, g, sm, s, dp);
        tile_logits(sm, g, n, j0, ks, s, x);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
            ds[a][bb] = b.sscale * exp2f(x[a][bb] - rL[a]) * (dp[a][bb] - rD[a]);
        __syncthreads();  // the band buffers become the dS tile
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) tA[(ty + 16 * a) * BN + tx + 16 * bb] = ds[a][bb];
        bucket_sums<true>(G, (size_t)H * R, n - i0, g, ds, far);
#pragma unroll
        for (int kc = 0; kc < D; kc += DC) {
          __syncthreads();
          stage_t<T, BN + 1>(gk + (size_t)(start + j0) * ts + (size_t)h * D + kc, ts, BN, n - j0, Ks);
          __syncthreads();
#pragma unroll 4
          for (int j = 0; j < BN; ++j) {
            const float k0 = Ks[tx * (BN + 1) + j], k1 = Ks[(tx + 16) * (BN + 1) + j];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const float d = tA[(ty + 16 * a) * BN + j];
              dq[a][kc / 16] = fmaf(d, k0, dq[a][kc / 16]);
              dq[a][kc / 16 + 1] = fmaf(d, k1, dq[a][kc / 16 + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = i0 + ty + 16 * a;
        // far-tile sums of the row: reduce over the 16 lanes that share it
#pragma unroll
        for (int sd = 0; sd < 2; ++sd)
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) far[a][sd] += __shfl_xor_sync(0xffffffffu, far[a][sd], off);
        if (i < n) {
          float* dst = b.dq + ((size_t)(start + i) * H + h) * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) dst[tx + 16 * c] = dq[a][c];
          if (tx == 0) {
            float* grow = G + (size_t)(ty + 16 * a) * H * R;
            if (far[a][0] != 0.f) atomicAdd(grow, far[a][0]);
            if (far[a][1] != 0.f) atomicAdd(grow + R - 1, far[a][1]);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ key side
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 2 : 1) bwd_k_kernel(const BwdProblem b) {
  extern __shared__ float sm[];
  const Problem& p = b.f;
  constexpr int NC = D / 16;
  const T* __restrict__ gq = static_cast<const T*>(p.q);
  const T* __restrict__ gdo = static_cast<const T*>(b.dout);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H, R = b.R;
  const size_t ts = (size_t)H * D;
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  float* tA = sm + BwdSmem::pk;  // P tile [BM][BN]
  float* tB = sm + BwdSmem::pq;  // dS tile [BM][BN]
  float* Qs = sm + BwdSmem::q;
  float* Gs = sm + BwdSmem::g;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 item = p.items[it];
    const int start = item.x, n = item.y, h = item.z, kb = item.w;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    const int nqb = (n + BM - 1) / BM;
    for (int sub = 0; sub < kQBlock / BN; ++sub) {
      const int j0 = kb * kQBlock + sub * BN;
      if (j0 >= n) break;
      float* G = b.gp + ((size_t)(start + j0) * H + h) * R;
      float dk[4][NC], dv[4][NC], far[4][2];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        far[a][0] = far[a][1] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) dk[a][c] = dv[a][c] = 0.f;
      }
      for (int ib = 0; ib < nqb; ++ib) {
        const int i0 = ib * BM;
        TileGeom g;
        tile_geom(p, rsp, rsn, i0, j0, ty, tx, g);
        float s[4][4], dp[4][4], x[4][4], pe[4][4], ds[4][4];
        score_tile<T, D, true>(p, gdo, scal_h, start, n, h, i0, j0, g, sm, s, dp);
        tile_logits(sm, g, n, j0, ks, s, x);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int i = i0 + ty + 16 * a;
          const size_t t = (size_t)start + i;
          const float rL = i < n ? b.lse[t * H + h] : INFINITY;
          const float rD = i < n ? b.drow[t * H + h] : 0.f;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            pe[a][bb] = exp2f(x[a][bb] - rL);
            ds[a][bb] = b.sscale * pe[a][bb] * (dp[a][bb] - rD);
          }
        }
        __syncthreads();  // the band buffers become the P and dS tiles
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            tA[(ty + 16 * a) * BN + tx + 16 * bb] = pe[a][bb];
            tB[(ty + 16 * a) * BN + tx + 16 * bb] = ds[a][bb];
          }
        bucket_sums<false>(G, (size_t)H * R, n - j0, g, ds, far);
        // dK += dS^T.Q and dV += P^T.dO over this query block, chunk by chunk;
        // thread rows are keys ty + 16 a
#pragma unroll
        for (int kc = 0; kc < D; kc += DC) {
          __syncthreads();
          const size_t qrow = (size_t)(start + i0) * ts + (size_t)h * D + kc;
          stage_t<T, BM + 1>(gq + qrow, ts, BM, n - i0, Qs);
          stage_t<T, BM + 1>(gdo + qrow, ts, BM, n - i0, Gs);
          __syncthreads();
#pragma unroll 4
          for (int i = 0; i < BM; ++i) {
            const float q0 = Qs[tx * (BM + 1) + i], q1 = Qs[(tx + 16) * (BM + 1) + i];
            const float g0 = Gs[tx * (BM + 1) + i], g1 = Gs[(tx + 16) * (BM + 1) + i];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const float sv = tB[i * BN + ty + 16 * a], pv = tA[i * BN + ty + 16 * a];
              dk[a][kc / 16] = fmaf(sv, q0, dk[a][kc / 16]);
              dk[a][kc / 16 + 1] = fmaf(sv, q1, dk[a][kc / 16 + 1]);
              dv[a][kc / 16] = fmaf(pv, g0, dv[a][kc / 16]);
              dv[a][kc / 16 + 1] = fmaf(pv, g1, dv[a][kc / 16 + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int j = j0 + ty + 16 * a;
        if (j < n) {
          const size_t row = ((size_t)(start + j) * H + h) * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            b.dk[row + tx + 16 * c] = dk[a][c];
            b.dv[row + tx + 16 * c] = dv[a][c];
          }
        }
      }
      // far-tile sums of key column tx + 16 u: the two half-warps hold
      // neighbouring query rows of the same keys
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int sd = 0; sd < 2; ++sd) {
          const float v = far[u][sd] + __shfl_xor_sync(0xffffffffu, far[u][sd], 16);
          const int jj = tx + 16 * u;
          if ((threadIdx.x & 16) == 0 && jj < n - j0 && v != 0.f)
            atomicAdd(G + (size_t)jj * H * R + (sd ? R - 1 : 0), v);
        }
    }
  }
}

// ------------------------------------------------------- strided fp32 GEMM
// C[s][b](m, n) (+)= sum over k in range s of A[b](m, k) B[b](k, n), every
// operand addressed by element strides; 64 x 64 tiles, k in steps of 16.
struct GemmArgs {
  const void* a;
  const void* b;
  float* c;
  long long sAb, sAm, sAk, sBb, sBk, sBn, sCs, sCb, sCm, sCn;
  int M, N, K, batch, kchunk, accumulate;
};

template <typename TA, typename TB>
__global__ void __launch_bounds__(256) gemm_kernel(const GemmArgs g) {
  __shared__ float As[16][64 + 1];
  __shared__ float Bs[16][64 + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int bb = blockIdx.z % g.batch, sp = blockIdx.z / g.batch;
  const int m0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
  const long long kb = (long long)sp * g.kchunk;
  const long long ke = min((long long)g.K, kb + g.kchunk);
  const TA* A = static_cast<const TA*>(g.a) + bb * g.sAb;
  const TB* B = static_cast<const TB*>(g.b) + bb * g.sBb;
  const bool a_kfast = g.sAk == 1, b_nfast = g.sBn == 1;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (long long k0 = kb; k0 < ke; k0 += 16) {
    __syncthreads();
    for (int e = tid; e < 16 * 64; e += 256) {
      const int ak = a_kfast ? e % 16 : e / 64, am = a_kfast ? e / 16 : e % 64;
      const long long k = k0 + ak;
      const int m = m0 + am;
      As[ak][am] = (k < ke && m < g.M) ? IO<TA>::load(A + m * g.sAm + k * g.sAk) : 0.f;
      const int bn = b_nfast ? e % 64 : e / 16, bk = b_nfast ? e / 64 : e % 16;
      const long long k2 = k0 + bk;
      const int nn = n0 + bn;
      Bs[bk][bn] = (k2 < ke && nn < g.N) ? IO<TB>::load(B + k2 * g.sBk + nn * g.sBn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  float* C = g.c + sp * g.sCs + bb * g.sCb;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty + 16 * i, nn = n0 + tx + 16 * j;
      if (m < g.M && nn < g.N) {
        float* dst = C + m * g.sCm + nn * g.sCn;
        *dst = g.accumulate ? *dst + acc[i][j] : acc[i][j];
      }
    }
}

// out[r][h][c] = sum over s of part[s][h][r][c]
__global__ void sum_splits_kernel(const float* __restrict__ part, int splits, int H, int R, int D,
                                  float* __restrict__ out) {
  const size_t total = (size_t)H * R * D;
  for (size_t f = (size_t)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (size_t)gridDim.x * blockDim.x) {
    const size_t h = f / ((size_t)R * D), r = (f / D) % R, c = f % D;
    float sum = 0.f;
    for (int s = 0; s < splits; ++s) sum += part[s * total + f];
    out[(r * H + h) * D + c] = sum;
  }
}

int num_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

template <typename TA, typename TB>
cudaError_t gemm(const GemmArgs& g, int splits, cudaStream_t s) {
  const dim3 grid((g.M + 63) / 64, (g.N + 63) / 64, g.batch * splits);
  gemm_kernel<TA, TB><<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_typed(const BwdProblem& b, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev_mid,
                         cudaEvent_t ev1, int* launches) {
  const Problem& p = b.f;
  const int H = p.H, R = b.R, T_ = p.T;
  const size_t bytes_q = BwdSmem::floats * sizeof(float);
  const size_t bytes_k = bytes_q;
  cudaError_t e = cudaFuncSetAttribute(bwd_q_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes_q);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_k_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes_k);
  if (e != cudaSuccess) return e;
  int occ_q = 0, occ_k = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_q, bwd_q_kernel<T, D>, kThreads, bytes_q);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_k, bwd_k_kernel<T, D>, kThreads, bytes_k);
  const int grid_q = std::min(p.max_items, num_sms() * std::max(occ_q, 1));
  const int grid_k = std::min(p.max_items, num_sms() * std::max(occ_k, 1));
  int n = 0;
  if (ev0) cudaEventRecord(ev0, s);
  if (grid_q > 0) {
    bwd_q_kernel<T, D><<<grid_q, kThreads, bytes_q, s>>>(b);
    ++n;
  }
  if (ev_mid) cudaEventRecord(ev_mid, s);
  if (grid_k > 0) {
    bwd_k_kernel<T, D><<<grid_k, kThreads, bytes_k, s>>>(b);
    ++n;
  }
  if (ev1) cudaEventRecord(ev1, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (T_ > 0) {
    const long long hd = (long long)H * D, hr = (long long)H * R;
    // dQ += G_c2p . PK and dK += G_p2c . PQ (per head: [T][R] x [R][d])
    GemmArgs g{};
    g.sAb = R; g.sAm = hr; g.sAk = 1;
    g.sBb = D; g.sBk = hd; g.sBn = 1;
    g.sCs = 0; g.sCb = D; g.sCm = hd; g.sCn = 1;
    g.M = T_; g.N = D; g.K = R; g.batch = H; g.kchunk = R; g.accumulate = 1;
    g.a = b.gc; g.b = p.pk; g.c = b.dq;
    if ((e = gemm<float, T>(g, 1, s)) != cudaSuccess) return e;
    g.a = b.gp; g.b = p.pq; g.c = b.dk;
    if ((e = gemm<float, T>(g, 1, s)) != cudaSuccess) return e;
    // partial dPK = G_c2p^T . Q and dPQ = G_p2c^T . K over token ranges
    GemmArgs r{};
    r.sAb = R; r.sAm = 1; r.sAk = hr;
    r.sBb = D; r.sBk = hd; r.sBn = 1;
    r.sCs = (long long)H * R * D; r.sCb = (long long)R * D; r.sCm = D; r.sCn = 1;
    r.M = R; r.N = D; r.K = T_; r.batch = H; r.kchunk = b.kchunk; r.accumulate = 0;
    r.a = b.gc; r.b = p.q; r.c = b.part;
    if ((e = gemm<float, T>(r, b.splits, s)) != cudaSuccess) return e;
    r.a = b.gp; r.b = p.k; r.c = b.part + (size_t)b.splits * H * R * D;
    if ((e = gemm<float, T>(r, b.splits, s)) != cudaSuccess) return e;
    const int blocks = std::min((H * R * D + 255) / 256, num_sms() * 8);
    sum_splits_kernel<<<blocks, 256, 0, s>>>(b.part, b.splits, H, R, D, b.dpk);
    sum_splits_kernel<<<blocks, 256, 0, s>>>(b.part + (size_t)b.splits * H * R * D, b.splits, H, R, D,
                                             b.dpq);
    n += 6;
  }
  *launches = n;
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const BwdProblem& b, cudaStream_t s, cudaEvent_t e0, cudaEvent_t em,
                         cudaEvent_t e1, int* n) {
  switch (b.f.d) {
    case 32: return launch_typed<T, 32>(b, s, e0, em, e1, n);
    case 64: return launch_typed<T, 64>(b, s, e0, em, e1, n);
    default: return launch_typed<T, 128>(b, s, e0, em, e1, n);
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem& b, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev_mid,
                       cudaEvent_t ev1, int* launches) {
  switch (b.f.dtype) {
    case DF_BF16: return launch_dtype<__nv_bfloat16>(b, s, ev0, ev_mid, ev1, launches);
    case DF_FP16: return launch_dtype<__half>(b, s, ev0, ev_mid, ev1, launches);
    default: return launch_dtype<float>(b, s, ev0, ev_mid, ev1, launches);
  }
}

}  // namespace dfa
