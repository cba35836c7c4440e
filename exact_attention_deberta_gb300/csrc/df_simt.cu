// Strict-FP32 fused forward on CUDA cores (FFMA, fp32 accumulation, no TF32).
//
// DisentangledFlash README, "Status", lists "strict FP32" next to the fast
// FP32/TF32 and FP16/BF16 modes.  This kernel is the strict one: every product
// and every sum is an IEEE fp32 operation.  It streams 64x64 score tiles with an
// online softmax (kernels-community "DisentangledFlash" discussion,
// "Motivation": tiled, streaming, exact) and never stores a score tile outside
// shared memory.
//
// Per tile the three logit terms are formed directly:
//   S   = Q_blk . K_blkᵀ                         (64 x 64 x d)
//   c2p = Q_i . PK[idx(i-j)],  p2c = K_j . PQ[idx(i-j)]
// For a near tile the PK / PQ rows of the tile's index band are staged in
// shared memory and each thread gathers, for its 4x4 micro-tile (rows ty+16a,
// columns tx+16b), the 7 band rows its diagonals touch.  A far tile lies
// entirely in a saturated part of the index table, so c2p and p2c are the
// per-token scalars prepared by the planning kernel.
#include "df_common.cuh"

#include <math.h>

#include <algorithm>

namespace dfa {

namespace {

constexpr int BM = 64;   // query rows per sub-block
constexpr int BN = 64;   // keys per tile
constexpr int DC = 32;   // head-dim chunk staged at once
constexpr int WB = 128;  // band capacity (BM + BN - 1 = 127 rows)
constexpr int kThreads = 256;

template <int D>
struct SimtSmem {
  static constexpr int q = DC * (BM + 1);
  static constexpr int k = DC * (BN + 1);
  static constexpr int band = DC * (WB + 1);
  static constexpr int v = BN * D;
  static constexpr int p = BM * (BN + 1);
  static constexpr int floats = q + k + 2 * band + v + p + 2 * BM + 3 * BN;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(Problem p) {
  extern __shared__ float smem[];
  using L = SimtSmem<D>;
  float* Qs = smem;               // [DC][BM+1]
  float* Ks = Qs + L::q;          // [DC][BN+1]
  float* PKs = Ks + L::k;         // [DC][WB+1]
  float* PQs = PKs + L::band;     // [DC][WB+1]
  float* Vs = PQs + L::band;      // [BN][D]
  float* Ps = Vs + L::v;          // [BM][BN+1]
  float* rowA = Ps + L::p;        // [2][BM]  alpha (neg side, pos side)
  float* colB = rowA + 2 * BM;    // [3][BN]  beta (neg, pos), key bias

  const T* __restrict__ gq = static_cast<const T*>(p.q);
  const T* __restrict__ gk = static_cast<const T*>(p.k);
  const T* __restrict__ gv = static_cast<const T*>(p.v);
  const T* __restrict__ gpk = static_cast<const T*>(p.pk);
  const T* __restrict__ gpq = static_cast<const T*>(p.pq);
  T* __restrict__ gout = static_cast<T*>(p.out);

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H;
  const size_t tok_stride = (size_t)H * D;
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  constexpr int NC = D / 16;  // output columns per thread

  // one work unit per 64-row half of an item: a small problem still fills
  // twice as many blocks
  constexpr int kSubs = kQBlock / BM;
  for (int u = blockIdx.x; u < n_items * kSubs; u += gridDim.x) {
    const int4 item = p.items[u / kSubs];
    const int start = item.x, n = item.y, h = item.z, qb = item.w;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    {
      const int sub = u % kSubs;
      const int i0 = qb * kQBlock + sub * BM;
      if (i0 >= n) continue;
      __syncthreads();
      for (int e = tid; e < BM; e += kThreads) {
        const int t = start + i0 + e;
        rowA[e] = i0 + e < n ? scal_h[0 * (size_t)p.t_pad + t] : 0.f;
        rowA[BM + e] = i0 + e < n ? scal_h[1 * (size_t)p.t_pad + t] : 0.f;
      }
      float m[4], l[4], o[4][NC];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) o[a][c] = 0.f;
      }
      const int nkb = (n + BN - 1) / BN;
      for (int jb = 0; jb < nkb; ++jb) {
        const int j0 = jb * BN;
        const int rlo = i0 - j0 - (BN - 1), rhi = i0 - j0 + (BM - 1);
        const bool far_pos = rlo >= rsp, far_neg = rhi <= rsn;
        const bool far = far_pos || far_neg;
        int lo = 0, w = 0;
        int col[7];
        if (!far) {
          lo = p.idx[rlo + p.lt - 1];
          w = p.idx[rhi + p.lt - 1] - lo + 1;
#pragma unroll
          for (int dd = 0; dd < 7; ++dd)
            col[dd] = p.idx[i0 - j0 + ty - tx + 16 * (dd - 3) + p.lt - 1] - lo;
        }
        __syncthreads();  // previous tile's Ps / Vs / colB readers are done
        for (int e = tid; e < BN; e += kThreads) {
          const int j = j0 + e;
          const int t = start + j;
          const bool ok = j < n;
          colB[e] = ok ? scal_h[2 * (size_t)p.t_pad + t] : -INFINITY;
          colB[BN + e] = ok ? scal_h[3 * (size_t)p.t_pad + t] : -INFINITY;
          colB[2 * BN + e] = ok ? p.keybias[t] : -INFINITY;
        }
        stage_rows<T, D, kThreads>(gv + (size_t)(start + j0) * tok_stride + (size_t)h * D, tok_stride, BN,
                                   n - j0, Vs);
        float s[4][4], cp[4][4], pc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) s[a][b] = cp[a][b] = pc[a][b] = 0.f;

        for (int kc = 0; kc < D; kc += DC) {
          if (kc) __syncthreads();
          const size_t hc = (size_t)h * D + kc;
          stage_transposed<T, DC, BM + 1, kThreads>(gq + (size_t)(start + i0) * tok_stride + hc, tok_stride,
                                                   BM, n - i0, Qs);
          stage_transposed<T, DC, BN + 1, kThreads>(gk + (size_t)(start + j0) * tok_stride + hc, tok_stride,
                                                   BN, n - j0, Ks);
          if (!far) {
            stage_transposed<T, DC, WB + 1, kThreads>(gpk + (size_t)lo * tok_stride + hc, tok_stride, w, w, PKs);
            stage_transposed<T, DC, WB + 1, kThreads>(gpq + (size_t)lo * tok_stride + hc, tok_stride, w, w, PQs);
          }
          __syncthreads();
          if (far) {
#pragma unroll 4
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
            }
          } else {
#pragma unroll 2
            for (int c = 0; c < DC; ++c) {
              float qa[4], kb[4], pkd[7], pqd[7];
#pragma unroll
              for (int a = 0; a < 4; ++a) qa[a] = Qs[c * (BM + 1) + ty + 16 * a];
#pragma unroll
              for (int b = 0; b < 4; ++b) kb[b] = Ks[c * (BN + 1) + tx + 16 * b];
#pragma unroll
              for (int dd = 0; dd < 7; ++dd) {
                pkd[dd] = PKs[c * (WB + 1) + col[dd]];
                pqd[dd] = PQs[c * (WB + 1) + col[dd]];
              }
#pragma unroll
              for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                  s[a][b] = fmaf(qa[a], kb[b], s[a][b]);
                  cp[a][b] = fmaf(qa[a], pkd[a - b + 3], cp[a][b]);
                  pc[a][b] = fmaf(kb[b], pqd[a - b + 3], pc[a][b]);
                }
            }
          }
        }

        // logits in log2 units, masked keys at -inf
        float x[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int jj = tx + 16 * b;
            float v;
            if (far) {
              const float al = far_pos ? rowA[BM + ty + 16 * a] : rowA[ty + 16 * a];
              const float be = far_pos ? colB[BN + jj] : colB[jj];
              v = fmaf(s[a][b], ks, al + be);
            } else {
              v = fmaf(s[a][b] + cp[a][b] + pc[a][b], ks, colB[2 * BN + jj]);
            }
            x[a][b] = j0 + jj < n ? v : -INFINITY;
          }
        // online softmax, row partials reduced over the 16 lanes sharing a row
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
          for (int b = 0; b < 4; ++b) {
            const float pv = exp2f(x[a][b] - base);
            l[a] += pv;
            Ps[(ty + 16 * a) * (BN + 1) + tx + 16 * b] = pv;
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
      // epilogue: normalise, write valid query rows (masked rows were zeroed by the planner)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float lt = l[a];
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        const int i = i0 + ty + 16 * a;
        if (i < n && p.keybias[start + i] == 0.f) {
          const float inv = 1.f / lt;
          T* dst = gout + (start + i) * tok_stride + (size_t)h * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) dst[tx + 16 * c] = IO<T>::from_f(o[a][c] * inv);
        }
      }
    }
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

template <typename T, int D>
cudaError_t launch_typed(const Problem& p, cudaStream_t s) {
  const size_t bytes = SimtSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.max_items * (kQBlock / BM), num_sms() * 2);
  if (grid <= 0) return cudaSuccess;
  simt_fwd_kernel<T, D><<<grid, kThreads, bytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const Problem& p, cudaStream_t s, int* launches) {
  *launches = p.max_items > 0 ? 1 : 0;
  switch (p.dtype) {
    case DF_BF16:
      return p.d == 32 ? launch_typed<__nv_bfloat16, 32>(p, s)
             : p.d == 64 ? launch_typed<__nv_bfloat16, 64>(p, s) : launch_typed<__nv_bfloat16, 128>(p, s);
    case DF_FP16:
      return p.d == 32 ? launch_typed<__half, 32>(p, s)
             : p.d == 64 ? launch_typed<__half, 64>(p, s) : launch_typed<__half, 128>(p, s);
    default:
      return p.d == 32 ? launch_typed<float, 32>(p, s)
             : p.d == 64 ? launch_typed<float, 64>(p, s) : launch_typed<float, 128>(p, s);
  }
}

}  // namespace dfa
