// Planning kernel: relative-position index table, varlen work list and the
// per-token position scalars used by far tiles.
//
// The index table is the DeBERTa log-bucketed relative position (DisentangledFlash
// README, "Status": C2P/P2C disentangled attention).  The work list realises the
// packed mode that never computes on padding (kernels-community "DisentangledFlash"
// discussion, the packed-vs-padded paragraph): a query block exists only for valid
// tokens, and sequences are ordered longest first so that a grid-stride loop over
// the list is a greedy longest-processing-time schedule.
#include "df_common.cuh"

#include <math.h>

namespace dfa {

namespace {

constexpr int kPlanThreads = 256;
constexpr int kScalarBlocks = 1216;  // 8 x 152 SMs, grid-stride over tokens

// ---- a1: one entry of the index table, plus the two saturation points -------
// r_sat_pos = smallest r with idx(r) = 2 span - 1, r_sat_neg = largest r with
// idx(r) = 0.  idx is non-decreasing in r, so each point has exactly one writer.
__device__ void index_entry(const Problem& p, int e) {
  const int lt = p.lt;
  const int r = e - (lt - 1);
  const int top = 2 * p.span - 1;
  const int u = rel_index(r, p.buckets, p.max_rel, p.span);
  p.idx[e] = u;
  if (u == top && (r == -(lt - 1) || rel_index(r - 1, p.buckets, p.max_rel, p.span) != top))
    p.hdr->r_sat_pos = r;
  if (r == lt - 1 && u != top) p.hdr->r_sat_pos = lt + kQBlock;  // never within reach
  if (u == 0 && (r == lt - 1 || rel_index(r + 1, p.buckets, p.max_rel, p.span) != 0))
    p.hdr->r_sat_neg = r;
  if (r == -(lt - 1) && u != 0) p.hdr->r_sat_neg = -(lt + kQBlock);
}

// ---- per-token position scalars (far tiles) and zeroing of padded rows -------
// scal[h][0..3][t] = kscale * {Q_t.PK[0], Q_t.PK[top], K_t.PQ[0], K_t.PQ[top]}.
// A masked (or out-of-range) key gets -inf in both K terms and in keybias.
template <typename T>
__device__ void scalar_token(const Problem& p, int t, int lane) {
  const int H = p.H, d = p.d, top = 2 * p.span - 1;
  const bool in_range = t < p.T;
  const bool valid = in_range && (p.packed || p.key_mask[t] != 0);
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* pk = static_cast<const T*>(p.pk);
  const T* pq = static_cast<const T*>(p.pq);
  if (lane == 0) p.keybias[t] = valid ? 0.f : -INFINITY;
  for (int h = 0; h < H; ++h) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (valid) {
      const size_t row = ((size_t)t * H + h) * d;
      for (int e = lane; e < d; e += 32) {
        const float qv = IO<T>::load(q + row + e);
        const float kv = IO<T>::load(k + row + e);
        a0 = fmaf(qv, IO<T>::load(pk + ((size_t)0 * H + h) * d + e), a0);
        a1 = fmaf(qv, IO<T>::load(pk + ((size_t)top * H + h) * d + e), a1);
        b0 = fmaf(kv, IO<T>::load(pq + ((size_t)0 * H + h) * d + e), b0);
        b1 = fmaf(kv, IO<T>::load(pq + ((size_t)top * H + h) * d + e), b1);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a0 += __shfl_xor_sync(0xffffffffu, a0, o);
        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
        b0 += __shfl_xor_sync(0xffffffffu, b0, o);
        b1 += __shfl_xor_sync(0xffffffffu, b1, o);
      }
    } else if (in_range) {
      T* out = static_cast<T*>(p.out) + ((size_t)t * H + h) * d;
      for (int e = lane; e < d; e += 32) out[e] = IO<T>::from_f(0.f);
    }
    if (lane == 0) {
      const size_t base = (size_t)h * 4 * p.t_pad + t;
      p.scal[base + 0 * (size_t)p.t_pad] = valid ? a0 * p.kscale : 0.f;
      p.scal[base + 1 * (size_t)p.t_pad] = valid ? a1 * p.kscale : 0.f;
      p.scal[base + 2 * (size_t)p.t_pad] = valid ? b0 * p.kscale : -INFINITY;
      p.scal[base + 3 * (size_t)p.t_pad] = valid ? b1 * p.kscale : -INFINITY;
    }
  }
}

// ---- a2: work list ------------------------------------------------------------
// One block.  For every sequence: start token, effective length n (packed: from
// cu_seqlens; padded: last valid position + 1) and nblk = ceil(n / 128).  Items
// {start, n, head, query block} are laid out sequence by sequence in
// non-increasing nblk order (ties keep the sequence order), head-major inside a
// sequence so that blocks sharing K/V run next to each other.
__device__ void build_worklist(const Problem& p) {
  const int B = p.B, L = p.L;
  // The status word reports the latest call: this block is the only one of the
  // planning kernel that can raise, so it clears the word before anything else.
  if (threadIdx.x == 0) { p.hdr->status = 0; p.hdr->status_where = 0; }
  __syncthreads();
  for (int s = threadIdx.x; s < B; s += blockDim.x) {
    int start, n;
    if (p.packed) {
      start = p.cu_seqlens[s];
      n = p.cu_seqlens[s + 1] - start;
      if (n < 0 || n > L || start < 0 || start + (n > 0 ? n : 0) > p.T) {
        raise_device_error(p.hdr, DF_ERR_INVALID_ARG, 100);
        n = 0;
      }
    } else {
      start = s * L;
      const uint8_t* row = p.key_mask + (size_t)s * L;
      n = 0;
      for (int j = L - 1; j >= 0; --j)
        if (row[j]) { n = j + 1; break; }
    }
    p.seqs[s] = make_int4(start, n, (n + kQBlock - 1) / kQBlock, 0);
  }
  __syncthreads();
  for (int s = threadIdx.x; s < B; s += blockDim.x) {
    const int4 me = p.seqs[s];
    int rank = 0, base = 0;
    for (int o = 0; o < B; ++o) {
      const int nb = p.seqs[o].z;
      const bool before = nb > me.z || (nb == me.z && o < s);
      rank += before;
      base += before ? nb * p.H : 0;
    }
    for (int h = 0; h < p.H; ++h)
      for (int b = 0; b < me.z; ++b)
        p.items[base + h * me.z + b] = make_int4(me.x, me.y, h, b);
    if (rank == B - 1) p.hdr->n_items = base + me.z * p.H;
    p.seqs[s].w = rank;
  }
  if (threadIdx.x == 0) {
    if (B == 0) p.hdr->n_items = 0;
    p.hdr->n_seqs = B;
  }
}

template <typename T>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Problem p, int nb_table) {
  const int bid = blockIdx.x;
  if (bid < nb_table) {
    const int e = bid * kPlanThreads + threadIdx.x;
    if (e < 2 * p.lt - 1) index_entry(p, e);
    return;
  }
  if (bid < nb_table + kScalarBlocks) {
    const int warp = (bid - nb_table) * (kPlanThreads / 32) + threadIdx.x / 32;
    const int nwarps = kScalarBlocks * (kPlanThreads / 32);
    for (int t = warp; t < p.t_pad; t += nwarps) scalar_token<T>(p, t, threadIdx.x & 31);
    return;
  }
  build_worklist(p);
}

__global__ void __launch_bounds__(kPlanThreads)
index_table_kernel(int buckets, int max_rel, int span, int max_len, int32_t* idx) {
  const int e = blockIdx.x * kPlanThreads + threadIdx.x;
  if (e < 2 * max_len - 1) idx[e] = rel_index(e - (max_len - 1), buckets, max_rel, span);
}

}  // namespace

cudaError_t launch_plan(const Problem& p, cudaStream_t s) {
  const int nb_table = (2 * p.lt - 1 + kPlanThreads - 1) / kPlanThreads;
  const int grid = nb_table + kScalarBlocks + 1;
  switch (p.dtype) {
    case DF_BF16: plan_kernel<__nv_bfloat16><<<grid, kPlanThreads, 0, s>>>(p, nb_table); break;
    case DF_FP16: plan_kernel<__half><<<grid, kPlanThreads, 0, s>>>(p, nb_table); break;
    default: plan_kernel<float><<<grid, kPlanThreads, 0, s>>>(p, nb_table); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_index_table(int buckets, int max_rel, int span, int max_len, int32_t* idx,
                               cudaStream_t s) {
  const int n = 2 * max_len - 1;
  index_table_kernel<<<(n + kPlanThreads - 1) / kPlanThreads, kPlanThreads, 0, s>>>(
      buckets, max_rel, span, max_len, idx);
  return cudaGetLastError();
}

}  // namespace dfa
