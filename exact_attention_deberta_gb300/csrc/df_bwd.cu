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
// Score tiles are 64 x 64 with 4 x 4 register micro-tiles (rows 4 ty + a,
// columns 4 tx + b, read as 16-byte vectors from swizzled shared buffers); the
// position terms of a near tile come from the PK / PQ rows of the tile's index
// band, and a far tile (every distance saturated) uses the per-token scalars of
// the planner.
#include "df_common.cuh"

#include <math.h>

#include <algorithm>

namespace dfa {

namespace {

constexpr int BM = 64;   // query rows per tile
constexpr int BN = 64;   // keys per tile
constexpr int DC = 32;   // head-dim chunk staged at once
constexpr int WB = 128;  // index-band capacity (BM + BN - 1 rows)
constexpr int CS = 68;   // row stride of the chunk and tile buffers (16-byte rows of 4)
constexpr int kThreads = 256;
static_assert(BM == BN, "query and key chunks are staged by one loop");

// Shared-memory map of the two tile kernels, in floats.  Thread (tx, ty) owns
// rows 4 ty + a and columns 4 tx + b of a tile, so its four operands of one
// step are one 16-byte load.
struct BwdSmem {
  static constexpr int q = 0;                      // [DC][CS] query chunk (swizzled rows)
  static constexpr int k = q + DC * CS;            // [DC][CS] key chunk
  static constexpr int g = k + DC * CS;            // [DC][CS] dO chunk
  static constexpr int v = g + DC * CS;            // [DC][CS] V chunk
  static constexpr int pk = v + DC * CS;           // [DC][WB + 1] PK band
  static constexpr int pq = pk + DC * (WB + 1);    // [DC][WB + 1] PQ band
  static constexpr int ta = pq + DC * (WB + 1);    // [BM][CS] dS tile (query side) / P tile (key side)
  static constexpr int tb = ta + BM * CS;          // [BM][CS] dS tile (key side)
  static constexpr int rowA = tb + BM * CS;        // [2][BM] query scalars (neg, pos side)
  static constexpr int colB = rowA + 2 * BM;       // [3][BN] key scalars (neg, pos), key bias
  static constexpr int floats = colB + 3 * BN;
  // pass 1 of the query kernel keeps V^T [D][CS] (swizzled like a chunk) in
  // the dO, V and band buffers, which it does not use after the scores, and P
  // [BM][CS] in tile A
  static constexpr int pass1 = g;
  static_assert(g + 128 * CS <= ta, "pass-1 V^T fits at d = 128");
  static_assert(q % 4 == 0 && k % 4 == 0 && g % 4 == 0 && v % 4 == 0 && ta % 4 == 0 && tb % 4 == 0,
                "16-byte aligned buffers");
};

// Row swizzle of the chunk buffers: row r of column c sits at r ^ swz(c).  The
// mask is a multiple of 4 below 32, so each group of four rows stays together
// and in order (16-byte reads), and the transposed 16-byte staging stores of a
// warp land in 32 different banks.
template <typename T>
__device__ __forceinline__ int swz(int c) {
  return (16 / (int)sizeof(T)) * ((c >> 3) & 3);
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

struct TileGeom {
  bool far_pos, far_neg, far;
  int lo, w;
  int col[7];  // band row of diagonal 4 (ty - tx) + dd - 3, relative to lo
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
    for (int dd = 0; dd < 7; ++dd) g.col[dd] = p.idx[i0 - j0 + 4 * (ty - tx) + dd - 3 + p.lt - 1] - g.lo;
  }
}

// dst[c * STRIDE + r'] = fp32 of row r, column c (c < DC) of a [rows][ts]
// array starting at `base`, for r < rows; rows at or past `lim` read as 0.
// SWZ: r' = r ^ swz(c) (chunk buffers), else r' = r (band buffers, odd
// stride).  Each thread moves 16-byte vectors.
template <typename T, int STRIDE, bool SWZ>
__device__ __forceinline__ void stage_t(const T* __restrict__ base, size_t ts, int rows, int lim,
                                        float* dst) {
  constexpr int V = 16 / sizeof(T);  // elements per vector
  constexpr int VPR = DC / V;        // vectors per row
  static_assert(SWZ || STRIDE % 32 == 1, "conflict-free transposed stores");
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
    for (int k = 0; k < V; ++k) {
      const int c = v * V + k;
      dst[c * STRIDE + (SWZ ? (r ^ swz<T>(c)) : r)] = f[k];
    }
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
    stage_t<T, CS, true>(gq + qrow, ts, BM, n - i0, Qs);
    stage_t<T, CS, true>(gk + krow, ts, BN, n - j0, Ks);
    if (DP) {
      stage_t<T, CS, true>(gdo + qrow, ts, BM, n - i0, Gs);
      stage_t<T, CS, true>(gv + krow, ts, BN, n - j0, Vc);
    }
    if (!g.far) {
      const size_t prow = (size_t)g.lo * ts + (size_t)h * D + kc;
      stage_t<T, WB + 1, false>(gpk + prow, ts, g.w, g.w, PKs);
      stage_t<T, WB + 1, false>(gpq + prow, ts, g.w, g.w, PQs);
    }
    __syncthreads();
#pragma unroll 2
    for (int c = 0; c < DC; ++c) {
      const int m = swz<T>(c);
      const float4 q4 = lds4(Qs + c * CS + ((4 * ty) ^ m));
      const float4 k4 = lds4(Ks + c * CS + ((4 * tx) ^ m));
      const float qa[4] = {q4.x, q4.y, q4.z, q4.w};
      const float kb[4] = {k4.x, k4.y, k4.z, k4.w};
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
        const float4 g4 = lds4(Gs + c * CS + ((4 * ty) ^ m));
        const float4 v4 = lds4(Vc + c * CS + ((4 * tx) ^ m));
        const float ga[4] = {g4.x, g4.y, g4.z, g4.w};
        const float vb[4] = {v4.x, v4.y, v4.z, v4.w};
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
      const int jj = 4 * tx + b;
      float v;
      if (g.far) {
        const float al = g.far_pos ? rowA[BM + 4 * ty + a] : rowA[4 * ty + a];
        const float be = g.far_pos ? colB[BN + jj] : colB[jj];
        v = fmaf(s[a][b], ks, al + be);
      } else {
        v = fmaf(s[a][b], ks, colB[2 * BN + jj]);
      }
      x[a][b] = j0 + jj < n ? v : -INFINITY;
    }
}

// Adds the tile's dS to the bucket sums.  G points at the table row of the
// block's first query row (BY_ROW) or key, rows `row_stride` floats apart;
// `lim` is the number of rows inside the sequence.  Near tiles add each
// nonzero entry to the global table; a far tile has one relative index
// (bucket 0 or 2 span - 1), so its entries go to the per-thread sums `far`
// ([row or column u][side]), flushed by the caller.
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
        const int row = BY_ROW ? 4 * ty + a : 4 * tx + b;
        if (row < lim && ds[a][b] != 0.f)
          atomicAdd(G + (size_t)row * row_stride + g.lo + g.col[a - b + 3], ds[a][b]);
      }
  }
}

// ---------------------------------------------------------------- query side
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) bwd_q_kernel(const BwdProblem b) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  const Problem& p = b.f;
  constexpr int NC = D / 16;  // output columns per thread: tx + 16 c
  const T* __restrict__ gk = static_cast<const T*>(p.k);
  const T* __restrict__ gv = static_cast<const T*>(p.v);
  const T* __restrict__ gdo = static_cast<const T*>(b.dout);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H, R = b.R;
  const size_t ts = (size_t)H * D;
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  float* Vt = sm + BwdSmem::pass1;  // pass 1: V^T [D][CS]
  float* tA = sm + BwdSmem::ta;     // pass 1: P tile, pass 2: dS tile [BM][CS]
  float* Ks = sm + BwdSmem::k;

  // one work unit per 64-row half of an item
  constexpr int kSubs = kQBlock / BM;
  for (int u = blockIdx.x; u < n_items * kSubs; u += gridDim.x) {
    const int4 item = p.items[u / kSubs];
    const int start = item.x, n = item.y, h = item.z, qb = item.w;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    const int nkb = (n + BN - 1) / BN;
    {
      const int i0 = qb * kQBlock + (u % kSubs) * BM;
      if (i0 >= n) continue;
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
        __syncthreads();  // V^T overwrites the band buffers
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
          float pv[4];
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            pv[bb] = exp2f(x[a][bb] - base);
            l[a] += pv[bb];
          }
          *reinterpret_cast<float4*>(tA + (4 * ty + a) * CS + 4 * tx) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        }
        // V^T of the key tile, column chunk by column chunk (the swizzle of a
        // column depends only on its position inside its chunk)
#pragma unroll
        for (int kc = 0; kc < D; kc += DC)
          stage_t<T, CS, true>(gv + (size_t)(start + j0) * ts + (size_t)h * D + kc, ts, BN, n - j0,
                               Vt + kc * CS);
        __syncthreads();
#pragma unroll 2
        for (int j = 0; j < BN; j += 4) {
          float4 p4[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) p4[a] = lds4(tA + (4 * ty + a) * CS + j);
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int col = tx + 16 * c;
            const float4 v4 = lds4(Vt + col * CS + (j ^ swz<T>(col)));
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              o[a][c] = fmaf(p4[a].x, v4.x, o[a][c]);
              o[a][c] = fmaf(p4[a].y, v4.y, o[a][c]);
              o[a][c] = fmaf(p4[a].z, v4.z, o[a][c]);
              o[a][c] = fmaf(p4[a].w, v4.w, o[a][c]);
            }
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
        const int i = i0 + 4 * ty + a;
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
        // the dS tile (its previous readers passed the barriers of score_tile)
#pragma unroll
        for (int a = 0; a < 4; ++a)
          *reinterpret_cast<float4*>(tA + (4 * ty + a) * CS + 4 * tx) =
              make_float4(ds[a][0], ds[a][1], ds[a][2], ds[a][3]);
        bucket_sums<true>(G, (size_t)H * R, n - i0, g, ds, far);
#pragma unroll
        for (int kc = 0; kc < D; kc += DC) {
          __syncthreads();
          stage_t<T, CS, true>(gk + (size_t)(start + j0) * ts + (size_t)h * D + kc, ts, BN, n - j0, Ks);
          __syncthreads();
          const int m0 = swz<T>(tx), m1 = swz<T>(tx + 16);
#pragma unroll 2
          for (int j = 0; j < BN; j += 4) {
            const float4 k0 = lds4(Ks + tx * CS + (j ^ m0));
            const float4 k1 = lds4(Ks + (tx + 16) * CS + (j ^ m1));
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const float4 d4 = lds4(tA + (4 * ty + a) * CS + j);
              float& q0 = dq[a][kc / 16];
              float& q1 = dq[a][kc / 16 + 1];
              q0 = fmaf(d4.x, k0.x, q0); q1 = fmaf(d4.x, k1.x, q1);
              q0 = fmaf(d4.y, k0.y, q0); q1 = fmaf(d4.y, k1.y, q1);
              q0 = fmaf(d4.z, k0.z, q0); q1 = fmaf(d4.z, k1.z, q1);
              q0 = fmaf(d4.w, k0.w, q0); q1 = fmaf(d4.w, k1.w, q1);
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = i0 + 4 * ty + a;
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
            float* grow = G + (size_t)(4 * ty + a) * H * R;
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
__global__ void __launch_bounds__(kThreads, 2) bwd_k_kernel(const BwdProblem b) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  const Problem& p = b.f;
  constexpr int NC = D / 16;  // output columns per thread: tx + 16 c
  const T* __restrict__ gq = static_cast<const T*>(p.q);
  const T* __restrict__ gdo = static_cast<const T*>(b.dout);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H, R = b.R;
  const size_t ts = (size_t)H * D;
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  float* tA = sm + BwdSmem::ta;  // P tile [BM][CS]
  float* tB = sm + BwdSmem::tb;  // dS tile [BM][CS]
  float* Qs = sm + BwdSmem::q;
  float* Gs = sm + BwdSmem::g;

  // one work unit per 64-key half of an item
  constexpr int kSubs = kQBlock / BN;
  for (int u = blockIdx.x; u < n_items * kSubs; u += gridDim.x) {
    const int4 item = p.items[u / kSubs];
    const int start = item.x, n = item.y, h = item.z, kb = item.w;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    const int nqb = (n + BM - 1) / BM;
    {
      const int j0 = kb * kQBlock + (u % kSubs) * BN;
      if (j0 >= n) continue;
      float* G = b.gp + ((size_t)(start + j0) * H + h) * R;
      // thread rows of dK / dV: keys 4 ty + a; columns tx + 16 c
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
          const int i = i0 + 4 * ty + a;
          const size_t t = (size_t)start + i;
          const float rL = i < n ? b.lse[t * H + h] : INFINITY;
          const float rD = i < n ? b.drow[t * H + h] : 0.f;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            pe[a][bb] = exp2f(x[a][bb] - rL);
            ds[a][bb] = b.sscale * pe[a][bb] * (dp[a][bb] - rD);
          }
        }
        // the P and dS tiles, by query row (their previous readers passed the
        // barriers of score_tile)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          *reinterpret_cast<float4*>(tA + (4 * ty + a) * CS + 4 * tx) =
              make_float4(pe[a][0], pe[a][1], pe[a][2], pe[a][3]);
          *reinterpret_cast<float4*>(tB + (4 * ty + a) * CS + 4 * tx) =
              make_float4(ds[a][0], ds[a][1], ds[a][2], ds[a][3]);
        }
        bucket_sums<false>(G, (size_t)H * R, n - j0, g, ds, far);
        // dK += dS^T.Q and dV += P^T.dO over this query block, chunk by chunk
#pragma unroll
        for (int kc = 0; kc < D; kc += DC) {
          __syncthreads();
          const size_t qrow = (size_t)(start + i0) * ts + (size_t)h * D + kc;
          stage_t<T, CS, true>(gq + qrow, ts, BM, n - i0, Qs);
          stage_t<T, CS, true>(gdo + qrow, ts, BM, n - i0, Gs);
          __syncthreads();
          const int m0 = swz<T>(tx), m1 = swz<T>(tx + 16);
#pragma unroll 2
          for (int i = 0; i < BM; i += 4) {
            const float4 q0 = lds4(Qs + tx * CS + (i ^ m0)), q1 = lds4(Qs + (tx + 16) * CS + (i ^ m1));
            const float4 g0 = lds4(Gs + tx * CS + (i ^ m0)), g1 = lds4(Gs + (tx + 16) * CS + (i ^ m1));
            const float qa0[4] = {q0.x, q0.y, q0.z, q0.w}, qa1[4] = {q1.x, q1.y, q1.z, q1.w};
            const float ga0[4] = {g0.x, g0.y, g0.z, g0.w}, ga1[4] = {g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float4 sv = lds4(tB + (i + u) * CS + 4 * ty);  // dS of query i + u, keys 4 ty..
              const float4 pv = lds4(tA + (i + u) * CS + 4 * ty);
              const float svs[4] = {sv.x, sv.y, sv.z, sv.w}, pvs[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
              for (int a = 0; a < 4; ++a) {
                dk[a][kc / 16] = fmaf(svs[a], qa0[u], dk[a][kc / 16]);
                dk[a][kc / 16 + 1] = fmaf(svs[a], qa1[u], dk[a][kc / 16 + 1]);
                dv[a][kc / 16] = fmaf(pvs[a], ga0[u], dv[a][kc / 16]);
                dv[a][kc / 16 + 1] = fmaf(pvs[a], ga1[u], dv[a][kc / 16 + 1]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int j = j0 + 4 * ty + a;
        if (j < n) {
          const size_t row = ((size_t)(start + j) * H + h) * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            b.dk[row + tx + 16 * c] = dk[a][c];
            b.dv[row + tx + 16 * c] = dv[a][c];
          }
        }
      }
      // far-tile sums of key column 4 tx + u: the two half-warps hold
      // neighbouring query rows of the same keys
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int sd = 0; sd < 2; ++sd) {
          const float v = far[u][sd] + __shfl_xor_sync(0xffffffffu, far[u][sd], 16);
          const int jj = 4 * tx + u;
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
  const int units = p.max_items * (kQBlock / BM);
  const int grid_q = std::min(units, num_sms() * std::max(occ_q, 1));
  const int grid_k = std::min(units, num_sms() * std::max(occ_k, 1));
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
