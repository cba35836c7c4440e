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

// ---- a1: the index table, plus the two saturation points ----------------------
// r_sat_pos = smallest r with idx(r) = 2 span - 1, r_sat_neg = largest r with
// idx(r) = 0.  idx is non-decreasing in r, so each point has exactly one writer.
// One warp per kTableRun = 30 consecutive entries: lane l evaluates entry
// base + l - 1, so that lanes 1..30 find both neighbours that the saturation
// tests compare with in the adjacent lanes, and lanes 0 and 31 only supply
// them.  Every lane evaluates exactly one double-precision bucket; GB300's
// FP64 pipe is slow, so the table is spread over many one-warp blocks rather
// than whole 256-thread blocks that would queue on a few SMs.
constexpr int kTableRun = 30;

__device__ void index_run(const Problem& p, int blk) {
  const int lane = threadIdx.x;
  if (lane >= 32) return;
  const int lt = p.lt, n = 2 * lt - 1, top = 2 * p.span - 1;
  const int e = blk * kTableRun + lane - 1;
  const int r = e - (lt - 1);
  const int u = rel_index(r, p.buckets, p.max_rel, p.span);
  const int prev = __shfl_up_sync(0xffffffffu, u, 1);    // idx(r - 1)
  const int next = __shfl_down_sync(0xffffffffu, u, 1);  // idx(r + 1)
  if (lane == 0 || lane == 31 || e >= n) return;
  p.idx[e] = u;
  if (u == top && (e == 0 || prev != top)) p.hdr->r_sat_pos = r;
  if (e == n - 1 && u != top) p.hdr->r_sat_pos = lt + kQBlock;  // never within reach
  if (u == 0 && (e == n - 1 || next != 0)) p.hdr->r_sat_neg = r;
  if (e == 0 && u != 0) p.hdr->r_sat_neg = -(lt + kQBlock);
}

// ---- per-token position scalars (far tiles) and zeroing of padded rows -------
// scal[h][0..3][t] = kscale * {Q_t.PK[0], Q_t.PK[top], K_t.PQ[0], K_t.PQ[top]}.
// A masked (or out-of-range) key gets -inf in both K terms and in keybias.
// One thread per (head, token); a block covers 256 tokens of one head and keeps
// that head's four position rows in shared memory.  A warp reads its 32 tokens'
// Q and K rows whole (a row's 16-byte pieces on consecutive lanes, so each load
// instruction covers whole rows), sums each row's products over its lanes and
// hands the four sums to the token's own thread.  The output rows of masked
// tokens (padded mode) are zeroed by each warp together, a whole row per group
// of lanes, so that every store fills whole 32-byte sectors.
template <typename T>
__device__ void scalar_block(const Problem& p, int blk) {
  __shared__ float rows[4][128];
  const int H = p.H, d = p.d, top = 2 * p.span - 1;
  const int tiles = (p.t_pad + kPlanThreads - 1) / kPlanThreads;
  const int h = blk / tiles;
  const int t = (blk % tiles) * kPlanThreads + threadIdx.x;
  const T* pk = static_cast<const T*>(p.pk);
  const T* pq = static_cast<const T*>(p.pq);
  const bool scal = p.scal_needed && !p.scal_in_near;
  for (int e = threadIdx.x; scal && e < 4 * d; e += kPlanThreads) {
    const int which = e / d, c = e % d;
    const T* src = which < 2 ? pk : pq;
    const int prow = (which & 1) ? top : 0;
    rows[which][c] = IO<T>::load(src + ((size_t)prow * H + h) * d + c);
  }
  __syncthreads();
  const bool in_range = t < p.T;
  const bool valid = in_range && (p.packed || p.key_mask[t] != 0);
  if (!p.packed && p.zero_out) {
    // the warp's 32 tokens (consecutive t, rows H * d elements apart): lanes
    // take consecutive 16-byte pieces of one row after another
    const int lane = threadIdx.x & 31;
    const unsigned zero = __ballot_sync(0xffffffffu, in_range && !valid);
    const int ppr = d * (int)sizeof(T) / 16;  // pieces per row: 4 .. 32
    const int t0 = t - lane;
    for (int e = lane; zero && e < 32 * ppr; e += 32) {
      const int r = e / ppr;
      if ((zero >> r) & 1u) {
        uint4* o4 = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)(t0 + r) * H + h) * d);
        o4[e % ppr] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  if (scal) {
    constexpr int kVec = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int ppr = d / kVec;   // 16-byte pieces per row: 8 .. 32, a power of two
    const int rpi = 32 / ppr;   // rows per load instruction
    const int c = lane % ppr;   // this lane's piece, the same in every row
    const int t0 = t - lane;
    float w[4][kVec];           // the piece of the four position rows
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < kVec; ++e) w[j][e] = rows[j][c * kVec + e];
    const unsigned live = __ballot_sync(0xffffffffu, valid);
    for (int it = 0; it < ppr; ++it) {
      const int r = it * rpi + lane / ppr;  // token t0 + r
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      if ((live >> r) & 1u) {
        const size_t off = ((size_t)(t0 + r) * H + h) * d + (size_t)c * kVec;
        const uint4 qv = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + off);
        const uint4 kv = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.k) + off);
        const T* qe = reinterpret_cast<const T*>(&qv);
        const T* ke = reinterpret_cast<const T*>(&kv);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const float qf = IO<T>::to_f(qe[e]), kf = IO<T>::to_f(ke[e]);
          s[0] = fmaf(qf, w[0][e], s[0]);
          s[1] = fmaf(qf, w[1][e], s[1]);
          s[2] = fmaf(kf, w[2][e], s[2]);
          s[3] = fmaf(kf, w[3][e], s[3]);
        }
      }
      for (int o = ppr / 2; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j], o);
      // token t0 + lane was summed in iteration lane / rpi by lanes
      // (lane % rpi) * ppr ..
      const int src = (lane % rpi) * ppr;
#pragma unroll
      for (int j = 0; j < 4; ++j) s[j] = __shfl_sync(0xffffffffu, s[j], src);
      if (lane / rpi == it) {
        a0 = s[0];
        a1 = s[1];
        b0 = s[2];
        b1 = s[3];
      }
    }
  }
  if (t >= p.t_pad) return;
  if (h == 0) p.keybias[t] = valid ? 0.f : -INFINITY;
  // No far tile at all (every sequence shorter than the saturation distance),
  // or the near-tile kernel forms the scalars and key-term blocks itself: only
  // the key bias (and the zeroed padded rows, above) remain.
  if (!scal) return;
  if constexpr (sizeof(T) == 2) {
    // key-term block of far tiles: raw p2c products as hi + lo, masked keys finite
    T v[16];
    const float c0 = valid ? b0 : kMaskedKeyTerm, c1 = valid ? b1 : kMaskedKeyTerm;
    const T h0 = IO<T>::from_f(c0), h1 = IO<T>::from_f(c1);
    v[0] = h0;
    v[1] = IO<T>::from_f(valid ? c0 - IO<T>::to_f(h0) : kMaskedKeyTerm);
    v[2] = h1;
    v[3] = IO<T>::from_f(valid ? c1 - IO<T>::to_f(h1) : kMaskedKeyTerm);
#pragma unroll
    for (int e = 4; e < 16; ++e) v[e] = IO<T>::from_f(0.f);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.kaug) + ((size_t)t * H + h) * 16);
    dst[0] = *reinterpret_cast<const uint4*>(v);
    dst[1] = *reinterpret_cast<const uint4*>(v + 8);
  }
  const size_t base = (size_t)h * 4 * p.t_pad + t;
  p.scal[base + 0 * (size_t)p.t_pad] = valid ? a0 * p.kscale : 0.f;
  p.scal[base + 1 * (size_t)p.t_pad] = valid ? a1 * p.kscale : 0.f;
  p.scal[base + 2 * (size_t)p.t_pad] = valid ? b0 * p.kscale : -INFINITY;
  p.scal[base + 3 * (size_t)p.t_pad] = valid ? b1 * p.kscale : -INFINITY;
}

// ---- a2: work list ------------------------------------------------------------
// One block.  For every sequence: start token, effective length n (packed: from
// cu_seqlens; padded: last valid position + 1) and nblk = ceil(n / 128).  Items
// {start, n, head, query block} are laid out sequence by sequence in
// non-increasing nblk order (ties keep the sequence order), head-major inside a
// sequence so that blocks sharing K/V run next to each other.
template <typename T>
__device__ void write_kaug_selectors(const Problem& p) {
  if constexpr (sizeof(T) == 2) {
    if (p.scal_in_near) {
      // per head: PK[0], PK[top], PQ[0], PQ[top], then twelve zero rows (d = 64)
      const int top = 2 * p.span - 1, H = p.H;
      T* dst = static_cast<T*>(p.absel);
      for (int e = threadIdx.x; e < H * 16 * 64; e += blockDim.x) {
        const int h = e / (16 * 64), row = (e / 64) % 16, c = e % 64;
        T v = IO<T>::from_f(0.f);
        if (row < 4) {
          const T* src = static_cast<const T*>(row < 2 ? p.pk : p.pq);
          v = src[((size_t)((row & 1) ? top : 0) * H + h) * 64 + c];
        }
        dst[e] = v;
      }
    }
    T* sel = static_cast<T*>(p.kaug_sel);
    for (int e = threadIdx.x; e < 256 * 16; e += blockDim.x) {
      const int row = e >> 4, c = e & 15;
      const bool one = row < 128 ? c < 2 : (c == 2 || c == 3);
      sel[e] = IO<T>::from_f(one ? 1.f : 0.f);
    }
  }
}

constexpr int kSmemSeqs = 512;  // batches up to this size rank in shared memory

__device__ void build_worklist(const Problem& p) {
  __shared__ int4 s_seq[kSmemSeqs];  // {start, n, nblk, first item}
  const int B = p.B, L = p.L;
  const bool in_smem = B <= kSmemSeqs;
  // The status word reports the latest call: this block is the only one of the
  // planning kernel that can raise, so it clears the word before anything else.
  if (threadIdx.x == 0) { p.hdr->status = 0; p.hdr->status_where = 0; p.hdr->next_item = 0; p.hdr->next_far_item = 0; }
  __syncthreads();
  if (p.packed) {
    for (int s = threadIdx.x; s < B; s += blockDim.x) {
      const int start = p.cu_seqlens[s];
      int n = p.cu_seqlens[s + 1] - start;
      if (n < 0 || n > L || start < 0 || start + (n > 0 ? n : 0) > p.T) {
        raise_device_error(p.hdr, DF_ERR_INVALID_ARG, 100);
        n = 0;
      }
      p.seqs[s] = make_int4(start, n, (n + kQBlock - 1) / kQBlock, 0);
      if (in_smem) s_seq[s] = p.seqs[s];
    }
  } else {
    // padded: n = last valid position + 1; one warp per batch row, each lane
    // takes every 32nd position and the warp keeps the largest valid one
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int s = threadIdx.x >> 5; s < B; s += nw) {
      const uint8_t* row = p.key_mask + (size_t)s * L;
      int last = -1;
      for (int j = lane; j < L; j += 32)
        if (row[j]) last = j;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      const int n = last + 1;
      if (lane == 0) {
        p.seqs[s] = make_int4(s * L, n, (n + kQBlock - 1) / kQBlock, 0);
        if (in_smem) s_seq[s] = p.seqs[s];
      }
    }
  }
  __syncthreads();
  for (int s = threadIdx.x; s < B; s += blockDim.x) {
    const int4 me = in_smem ? s_seq[s] : p.seqs[s];
    int rank = 0, base = 0;
    for (int o = 0; o < B; ++o) {
      const int nb = in_smem ? s_seq[o].z : p.seqs[o].z;
      const bool before = nb > me.z || (nb == me.z && o < s);
      rank += before;
      base += before ? nb * p.H : 0;
    }
    if (!in_smem)
      for (int h = 0; h < p.H; ++h)
        for (int b = 0; b < me.z; ++b)
          p.items[base + h * me.z + b] = make_int4(me.x, me.y, h, b);
    if (rank == B - 1) p.hdr->n_items = base + me.z * p.H;
    p.seqs[s].w = rank;
    if (in_smem) s_seq[s].w = base;  // read back only after the barrier below
  }
  if (in_smem) {
    // the whole block writes every sequence's items
    __syncthreads();
    for (int s = 0; s < B; ++s) {
      const int4 me = s_seq[s];
      const int count = me.z * p.H;
      for (int e = threadIdx.x; e < count; e += blockDim.x)
        p.items[me.w + e] = make_int4(me.x, me.y, e / me.z, e % me.z);
    }
  }
  if (threadIdx.x == 0) {
    if (B == 0) p.hdr->n_items = 0;
    p.hdr->n_seqs = B;
  }
}

// ---- diagonal position tables (near tiles of the 16-bit tensor-core kernels) ----
// Row r of each table is the PK (PQ) row at idx(128 diag_m0 - 127 + r), for r in
// [0, 128 (n_diag + 1)): the 256 diagonals t of tile offset m are rows
// 128 (m - diag_m0) + t, so that neighbouring offsets share half their rows.
// With them the position products of a near tile come out of the MMA already
// indexed by diagonal.  A block copies kDiagRows rows of one table in 16-byte
// pieces; their source rows are looked up once.
constexpr int kDiagRows = 8;

__device__ void diag_rows(const Problem& p, int blk) {
  __shared__ int src_row[kDiagRows];
  const int cpr = p.H * p.d * 2 / 16;  // 16-byte pieces per row (16-bit types)
  const int rows = (p.n_diag + 1) * 128;
  const int which = blk / (rows / kDiagRows);
  const int row0 = (blk % (rows / kDiagRows)) * kDiagRows;
  if (threadIdx.x < kDiagRows) {
    const int row = row0 + threadIdx.x;
    src_row[threadIdx.x] = rel_index(128 * p.diag_m0 - 127 + row, p.buckets, p.max_rel, p.span);
  }
  __syncthreads();
  const uint4* src = static_cast<const uint4*>(which ? p.pq : p.pk);
  uint4* dst = static_cast<uint4*>(which ? p.diag_pq : p.diag_pk);
  for (int e = threadIdx.x; e < kDiagRows * cpr; e += kPlanThreads) {
    const int r = e / cpr, c = e % cpr;
    dst[(size_t)(row0 + r) * cpr + c] = src[(size_t)src_row[r] * cpr + c];
  }
}

template <typename T>
__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(Problem p, int nb_table, int nb_scal, int nb_diag) {
  allow_dependent_launch();  // the attention kernel waits for this grid's end
  if (blockIdx.x == 0) {  // the single work-list block starts first
    write_kaug_selectors<T>(p);
    build_worklist(p);
    return;
  }
  const int bid = blockIdx.x - 1;
  if (bid < nb_table) {
    index_run(p, bid);
    return;
  }
  if (bid < nb_table + nb_scal) {
    scalar_block<T>(p, bid - nb_table);
    return;
  }
  diag_rows(p, bid - nb_table - nb_scal);
}

__global__ void __launch_bounds__(kPlanThreads)
index_table_kernel(int buckets, int max_rel, int span, int max_len, int32_t* idx) {
  const int e = blockIdx.x * kPlanThreads + threadIdx.x;
  if (e < 2 * max_len - 1) idx[e] = rel_index(e - (max_len - 1), buckets, max_rel, span);
}

}  // namespace

cudaError_t launch_plan(const Problem& p, cudaStream_t s) {
  const int nb_table = (2 * p.lt - 1 + kTableRun - 1) / kTableRun;
  const int nb_scal = p.H * ((p.t_pad + kPlanThreads - 1) / kPlanThreads);
  // diagonal tables: 16-bit I/O types only (the strict-fp32 kernel does not use them)
  const int nb_diag = p.dtype == DF_FP32 || p.n_diag < 1 ? 0 : 2 * (p.n_diag + 1) * 128 / kDiagRows;
  const int grid = nb_table + nb_scal + nb_diag + 1;
  switch (p.dtype) {
    case DF_BF16:
      plan_kernel<__nv_bfloat16><<<grid, kPlanThreads, 0, s>>>(p, nb_table, nb_scal, nb_diag);
      break;
    case DF_FP16:
      plan_kernel<__half><<<grid, kPlanThreads, 0, s>>>(p, nb_table, nb_scal, nb_diag);
      break;
    default: plan_kernel<float><<<grid, kPlanThreads, 0, s>>>(p, nb_table, nb_scal, nb_diag); break;
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
