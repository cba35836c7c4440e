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
// Each thread owns a 4x4 micro-tile (rows ty + 16 a, keys tx + 16 b).  For a
// near tile the PK / PQ rows of the tile's index band are staged in shared
// memory and each thread reads, for its micro-tile, the 7 band rows its
// diagonals touch.  A far tile lies entirely in a saturated part of the index
// table, so c2p and p2c are the per-token scalars of the planning kernel.
//
// Shared memory holds every operand row-major, as in global memory, so that
// the copies are plain 16-byte cp.async transfers, and the FFMA loops read
// 16-byte vectors of four consecutive head-dimension (or key) elements: one
// vector load feeds four FMAs per operand pair.  Row strides of 4 (mod 8)
// words keep the eight lanes of each 16-byte load phase in distinct banks.
// The query rows of a work unit stay resident; the key rows and band rows of
// the next 32-column chunk are copied while the current one is multiplied
// (two buffers), and the next tile's V while the current tile's softmax and
// P.V run.
#include "df_common.cuh"

#include <math.h>

#include <algorithm>

namespace dfa {

namespace {

constexpr int BM = 64;   // query rows per work unit
constexpr int BN = 64;   // keys per tile
constexpr int DC = 32;   // head-dimension chunk staged at once
constexpr int WB = 128;  // band capacity (BM + BN - 1 = 127 rows)
constexpr int kThreads = 256;
constexpr int SC = DC + 4;  // row stride (words) of the key and band chunks
constexpr int SP = BN + 4;  // row stride of P

template <int D>
struct SimtSmem {
  static constexpr int SQ = D + 4;  // row stride of Q and V
  static constexpr int q = 0;                      // [BM][SQ]
  static constexpr int v = q + BM * SQ;            // [BN][SQ]
  static constexpr int p = v + BN * SQ;            // [BM][SP]
  static constexpr int stage = p + BM * SP;        // [2][K chunk | PK band | PQ band]
  static constexpr int k_off = 0, pk_off = BN * SC, pq_off = pk_off + WB * SC;
  static constexpr int stage_floats = pq_off + WB * SC;
  static constexpr int floats = stage + 2 * stage_floats;
  static constexpr size_t bytes = floats * sizeof(float);
  static_assert((SQ / 4) % 2 == 1 && (SC / 4) % 2 == 1 && (SP / 4) % 2 == 1,
                "odd 16-byte strides: conflict-free vector loads");
  static_assert(v % 4 == 0 && p % 4 == 0 && stage % 4 == 0 && stage_floats % 4 == 0,
                "16-byte aligned regions");
};

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp16(float* dst, const float* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) simt_fwd_kernel(Problem p) {
  extern __shared__ __align__(16) float smem[];
  using L = SimtSmem<D>;
  constexpr int SQ = L::SQ;
  constexpr int NCH = D / DC;  // chunks per tile
  static_assert(D % DC == 0, "whole chunks");
  float* Qs = smem + L::q;
  float* Vs = smem + L::v;
  float* Ps = smem + L::p;
  float* stage0 = smem + L::stage;

  const float* __restrict__ gq = static_cast<const float*>(p.q);
  const float* __restrict__ gk = static_cast<const float*>(p.k);
  const float* __restrict__ gv = static_cast<const float*>(p.v);
  const float* __restrict__ gpk = static_cast<const float*>(p.pk);
  const float* __restrict__ gpq = static_cast<const float*>(p.pq);
  float* __restrict__ gout = static_cast<float*>(p.out);

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = p.H;
  const size_t tok_stride = (size_t)H * D;
  grid_dependency_wait();  // the planner's outputs (first global access below)
  const int n_items = p.hdr->n_items;
  const int rsp = p.hdr->r_sat_pos, rsn = p.hdr->r_sat_neg;
  const float ks = p.kscale;
  // output columns of this thread: 4 tx + c + 64 m (d >= 64), 2 tx + c (d = 32)
  constexpr int CW = D >= 64 ? 4 : 2;    // consecutive columns per group
  constexpr int NG = D >= 64 ? D / 64 : 1;  // column groups
  constexpr int NC = CW * NG;

  // one work unit per 64-row half of an item: a small problem still fills
  // twice as many blocks
  constexpr int kSubs = kQBlock / BM;
  for (int u = blockIdx.x; u < n_items * kSubs; u += gridDim.x) {
    const int4 item = p.items[u / kSubs];
    const int start = item.x, n = item.y, h = item.z, qb = item.w;
    const int i0 = qb * kQBlock + (u % kSubs) * BM;
    if (i0 >= n) continue;
    const float* scal_h = p.scal + (size_t)h * 4 * p.t_pad;
    const int nkb = (n + BN - 1) / BN;
    const int n_stages = nkb * NCH;

    // tile geometry: far (and on which side) or the band [lo, lo + w) of PK / PQ
    auto tile_far = [&](int jb, bool* pos) {
      const int j0 = jb * BN;
      const int rlo = i0 - j0 - (BN - 1), rhi = i0 - j0 + (BM - 1);
      *pos = rlo >= rsp;
      return rlo >= rsp || rhi <= rsn;
    };
    // copies of stage s: the key rows and (near tiles) band rows of its chunk
    auto issue_stage = [&](int s) {
      const int jb = s / NCH, kc = (s % NCH) * DC, j0 = jb * BN;
      float* st = stage0 + (s & 1) * L::stage_floats;
      for (int e = tid; e < BN * (DC / 4); e += kThreads) {
        const int r = e / (DC / 4), c = 4 * (e % (DC / 4));
        const bool ok = j0 + r < n;
        cp16(st + L::k_off + r * SC + c, ok ? gk + (size_t)(start + j0 + r) * tok_stride + h * D + kc + c : gk,
             ok ? 16 : 0);
      }
      bool pos;
      if (!tile_far(jb, &pos)) {
        const int lo = p.idx[i0 - j0 - (BN - 1) + p.lt - 1];
        const int w = p.idx[i0 - j0 + (BM - 1) + p.lt - 1] - lo + 1;
        for (int e = tid; e < 2 * w * (DC / 4); e += kThreads) {
          const int which = e / (w * (DC / 4)), f = e % (w * (DC / 4));
          const int r = f / (DC / 4), c = 4 * (f % (DC / 4));
          const float* src = (which ? gpq : gpk) + (size_t)(lo + r) * tok_stride + h * D + kc + c;
          cp16(st + (which ? L::pq_off : L::pk_off) + r * SC + c, src, 16);
        }
      }
    };
    auto issue_v = [&](int jb) {
      const int j0 = jb * BN;
      for (int e = tid; e < BN * (D / 4); e += kThreads) {
        const int r = e / (D / 4), c = 4 * (e % (D / 4));
        const bool ok = j0 + r < n;
        cp16(Vs + r * SQ + c, ok ? gv + (size_t)(start + j0 + r) * tok_stride + h * D + c : gv, ok ? 16 : 0);
      }
    };

    __syncthreads();  // the previous unit's readers of Q, V, P and the stages are done
    for (int e = tid; e < BM * (D / 4); e += kThreads) {
      const int r = e / (D / 4), c = 4 * (e % (D / 4));
      const bool ok = i0 + r < n;
      cp16(Qs + r * SQ + c, ok ? gq + (size_t)(start + i0 + r) * tok_stride + h * D + c : gq, ok ? 16 : 0);
    }
    issue_v(0);
    issue_stage(0);
    cp_commit();

    float a_neg[4], a_pos[4];  // this thread's rows: Q.PK[0] and Q.PK[top] (log2 units)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + ty + 16 * a;
      a_neg[a] = i < n ? scal_h[start + i] : 0.f;
      a_pos[a] = i < n ? scal_h[(size_t)p.t_pad + start + i] : 0.f;
    }
    float m[4], l[4], o[4][NC];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      m[a] = -INFINITY;
      l[a] = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) o[a][c] = 0.f;
    }
    float s[4][4], cp[4][4], pc[4][4];
    int col[7];
    bool far = false, far_pos = false;

    for (int st_i = 0; st_i < n_stages; ++st_i) {
      const int jb = st_i / NCH, kc = (st_i % NCH) * DC, j0 = jb * BN;
      if (kc == 0) {
        far = tile_far(jb, &far_pos);
        if (!far) {
          const int lo = p.idx[i0 - j0 - (BN - 1) + p.lt - 1];
#pragma unroll
          for (int dd = 0; dd < 7; ++dd)
            col[dd] = p.idx[i0 - j0 + ty - tx + 16 * (dd - 3) + p.lt - 1] - lo;
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) s[a][b] = cp[a][b] = pc[a][b] = 0.f;
      }
      // the next stage's copies go out before this one is awaited
      if (st_i + 1 < n_stages) {
        issue_stage(st_i + 1);
        cp_commit();
        cp_wait<1>();
      } else {
        cp_wait<0>();
      }
      __syncthreads();
      const float* st = stage0 + (st_i & 1) * L::stage_floats;
      const float* kst = st + L::k_off;
      const float* pkst = st + L::pk_off;
      const float* pqst = st + L::pq_off;
#pragma unroll 2
      for (int c4 = 0; c4 < DC; c4 += 4) {
        float4 qa[4], kb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) qa[a] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * a) * SQ + kc + c4);
#pragma unroll
        for (int b = 0; b < 4; ++b) kb[b] = *reinterpret_cast<const float4*>(kst + (tx + 16 * b) * SC + c4);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            s[a][b] = fmaf(qa[a].x, kb[b].x, s[a][b]);
            s[a][b] = fmaf(qa[a].y, kb[b].y, s[a][b]);
            s[a][b] = fmaf(qa[a].z, kb[b].z, s[a][b]);
            s[a][b] = fmaf(qa[a].w, kb[b].w, s[a][b]);
          }
        if (!far) {
          float4 bd[7];
#pragma unroll
          for (int dd = 0; dd < 7; ++dd) bd[dd] = *reinterpret_cast<const float4*>(pkst + col[dd] * SC + c4);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float4 e = bd[a - b + 3];
              cp[a][b] = fmaf(qa[a].x, e.x, cp[a][b]);
              cp[a][b] = fmaf(qa[a].y, e.y, cp[a][b]);
              cp[a][b] = fmaf(qa[a].z, e.z, cp[a][b]);
              cp[a][b] = fmaf(qa[a].w, e.w, cp[a][b]);
            }
#pragma unroll
          for (int dd = 0; dd < 7; ++dd) bd[dd] = *reinterpret_cast<const float4*>(pqst + col[dd] * SC + c4);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float4 e = bd[a - b + 3];
              pc[a][b] = fmaf(kb[b].x, e.x, pc[a][b]);
              pc[a][b] = fmaf(kb[b].y, e.y, pc[a][b]);
              pc[a][b] = fmaf(kb[b].z, e.z, pc[a][b]);
              pc[a][b] = fmaf(kb[b].w, e.w, pc[a][b]);
            }
        }
      }
      if (kc + DC < D) {
        __syncthreads();  // this stage's buffer takes stage st_i + 2
        continue;
      }

      // ---- the tile is complete: logits in log2 units, masked keys at -inf
      float x[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int j = j0 + tx + 16 * b;
        const bool ok = j < n;
        const size_t t = (size_t)start + j;
        // key terms of this column: far tiles take the saturated p2c scalar,
        // near tiles the key bias (0, or -inf for a masked key)
        const float kterm = !ok ? -INFINITY
                                : far ? scal_h[(far_pos ? 3 : 2) * (size_t)p.t_pad + t] : p.keybias[t];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float v = far ? fmaf(s[a][b], ks, (far_pos ? a_pos[a] : a_neg[a]) + kterm)
                              : fmaf(s[a][b] + cp[a][b] + pc[a][b], ks, kterm);
          x[a][b] = ok ? v : -INFINITY;
        }
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
          Ps[(ty + 16 * a) * SP + tx + 16 * b] = pv;
        }
      }
      __syncthreads();  // P stored; every thread is done with this tile's stage buffers
#pragma unroll 2
      for (int j4 = 0; j4 < BN; j4 += 4) {
        float4 pa[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) pa[a] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * a) * SP + j4);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float vv[NC];
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            if constexpr (CW == 4) {
              const float4 t4 = *reinterpret_cast<const float4*>(Vs + (j4 + jj) * SQ + 64 * g + 4 * tx);
              vv[4 * g] = t4.x;
              vv[4 * g + 1] = t4.y;
              vv[4 * g + 2] = t4.z;
              vv[4 * g + 3] = t4.w;
            } else {
              const float2 t2 = *reinterpret_cast<const float2*>(Vs + (j4 + jj) * SQ + 2 * tx);
              vv[0] = t2.x;
              vv[1] = t2.y;
            }
          }
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float pj = jj == 0 ? pa[a].x : jj == 1 ? pa[a].y : jj == 2 ? pa[a].z : pa[a].w;
#pragma unroll
            for (int c = 0; c < NC; ++c) o[a][c] = fmaf(pj, vv[c], o[a][c]);
          }
        }
      }
      __syncthreads();  // P and V are free
      if (jb + 1 < nkb) {
        issue_v(jb + 1);
        cp_commit();
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
        float* dst = gout + (start + i) * tok_stride + (size_t)h * D;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          if constexpr (CW == 4)
            *reinterpret_cast<float4*>(dst + 64 * g + 4 * tx) =
                make_float4(o[a][4 * g] * inv, o[a][4 * g + 1] * inv, o[a][4 * g + 2] * inv, o[a][4 * g + 3] * inv);
          else
            *reinterpret_cast<float2*>(dst + 2 * tx) = make_float2(o[a][0] * inv, o[a][1] * inv);
        }
      }
    }
  }
  cp_wait<0>();  // no copy may still be landing when the CTA leaves
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

template <int D>
cudaError_t launch_typed(const Problem& p, cudaStream_t s) {
  const size_t bytes = SimtSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.max_items * (kQBlock / BM), num_sms());
  if (grid <= 0) return cudaSuccess;
  e = launch_after_plan(simt_fwd_kernel<D>, grid, kThreads, bytes, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// fp32 I/O only: 16-bit inputs take the tensor-core kernels.
cudaError_t launch_simt(const Problem& p, cudaStream_t s, int* launches) {
  *launches = p.max_items > 0 ? 1 : 0;
  if (p.dtype != DF_FP32) return cudaErrorInvalidValue;
  return p.d == 32 ? launch_typed<32>(p, s) : p.d == 64 ? launch_typed<64>(p, s) : launch_typed<128>(p, s);
}

}  // namespace dfa
