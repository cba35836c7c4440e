// Host side of the C ABI declared in include/df_attn.h: argument checks,
// workspace layout, planning launch and dispatch to the fused kernels.
//
// Error policy follows the strict-contract convention of the pages' prior art
// (FastFlashAttention README, "API": an unsupported configuration is an error,
// never a hidden slow path): every check runs before the first launch and a
// failing one returns a status with nothing enqueued.
#include "df_common.cuh"

#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

namespace dfa {
cudaError_t launch_tc(const Problem& p, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev_mid,
                      cudaEvent_t ev1, int* launches);
bool tc_enabled();
}  // namespace dfa

namespace {

using namespace dfa;

std::atomic<unsigned long long> g_wait_budget{0};
cudaEvent_t g_prof_start = nullptr;
cudaEvent_t g_prof_stop = nullptr;
cudaEvent_t g_prof_mid = nullptr;
std::atomic<int> g_last_launches{0};

constexpr unsigned long long kDefaultWaitBudget = 1ull << 31;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t header, idx, items, seqs, scal, keybias, partial, diag_pk, diag_pq, kaug, kaug_sel, absel,
      total;
  int max_items, t_pad, lt, n_diag, diag_m0;
};

// Host copy of the bucket function (double precision, as on the device); used
// only to size the diagonal tables.
int host_rel_index(int r, int buckets, int max_rel, int span) {
  int b = r;
  if (buckets > 0) {
    const int mid = buckets / 2;
    const int a = r < 0 ? -r : r;
    if (a > mid) {
      const double f = log((double)a / (double)mid) / log((double)(max_rel - 1) / (double)mid);
      const int g = (int)ceil(f * (double)(mid - 1)) + mid;
      b = r < 0 ? -g : g;
    }
  }
  const int u = b + span;
  return u < 0 ? 0 : (u > 2 * span - 1 ? 2 * span - 1 : u);
}

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Saturation points of the bucket function within |r| < lt: rsp = the smallest
// r >= 0 with idx(r) = 2 span - 1 (lt + 128 if there is none), rsn = the largest
// r <= 0 with idx(r) = 0 (-(lt + 128) if none).  Finding them scans up to lt
// double-precision buckets per side, tens of microseconds of host time, so the
// last few parameter sets a process used are kept (the result depends on
// nothing else).
struct SatPoints {
  int rsp, rsn;
};

SatPoints saturation_points(int buckets, int max_rel, int span, int lt) {
  struct Entry {
    int buckets, max_rel, span, lt;
    SatPoints s;
  };
  constexpr int kKept = 8;
  static std::mutex mu;
  static Entry kept[kKept];
  static int n_kept = 0, next = 0;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n_kept; ++i) {
      const Entry& e = kept[i];
      if (e.buckets == buckets && e.max_rel == max_rel && e.span == span && e.lt == lt) return e.s;
    }
  }
  const int top = 2 * span - 1;
  SatPoints s{lt + kQBlock, -(lt + kQBlock)};
  for (int r = 0; r < lt; ++r)
    if (host_rel_index(r, buckets, max_rel, span) == top) { s.rsp = r; break; }
  for (int r = 0; r > -lt; --r)
    if (host_rel_index(r, buckets, max_rel, span) == 0) { s.rsn = r; break; }
  std::lock_guard<std::mutex> g(mu);
  kept[next] = Entry{buckets, max_rel, span, lt, s};
  next = (next + 1) % kKept;
  if (n_kept < kKept) ++n_kept;
  return s;
}

// Tile offsets m = query block - key block that can hold a near tile: the tile's
// distances [128 m - 127, 128 m + 127] are not all saturated.  One offset of
// slack on each side absorbs a last-ulp difference between host and device logs.
void near_offsets(int L, int buckets, int max_rel, int span, int lt, int* m0, int* n) {
  const SatPoints sat = saturation_points(buckets, max_rel, span, lt);
  const int rsp = sat.rsp, rsn = sat.rsn;
  const int nkb = (L + kKBlock - 1) / kKBlock;
  // strict range: floor((rsn - 127) / 128) + 1 .. ceil((rsp + 127) / 128) - 1
  int lo = floor_div(rsn - 127, 128);
  int hi = -floor_div(-(rsp + 127), 128);
  lo = lo < -(nkb - 1) ? -(nkb - 1) : lo;
  hi = hi > nkb - 1 ? nkb - 1 : hi;
  *m0 = lo;
  *n = hi >= lo ? hi - lo + 1 : 0;
}

// Whether a far tile (every distance of a 128 x 128 tile saturated) can occur
// for sequences of at most L tokens.  The largest offset is 128 (nkb - 1); a
// margin of 2 in r covers a last-ulp difference between host and device logs,
// so "no" here is "no" on the device too.
// Whether a tile of `tile` queries x `tile` keys of some sequence (length <= L)
// can lie wholly beyond a saturation point (a far tile).
bool far_tiles_possible(int L, int buckets, int max_rel, int span, int lt, int tile) {
  const SatPoints sat = saturation_points(buckets, max_rel, span, lt);
  const int rsp = sat.rsp, rsn = sat.rsn;
  const int reach = tile * ((L + tile - 1) / tile - 1) - (tile - 1);
  return reach >= rsp - 2 || -reach <= rsn + 2;
}

Layout make_layout(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  Layout l{};
  l.lt = ((L + 127) / 128) * 128 + 128;
  const size_t T = (size_t)B * L;
  l.t_pad = (int)(((T + 128 + 127) / 128) * 128);
  l.max_items = B * H * ((L + kQBlock - 1) / kQBlock);
  size_t off = 0;
  l.header = off;
  off = align256(off + sizeof(df_ws_header));
  l.idx = off;
  off = align256(off + (size_t)(2 * l.lt - 1) * sizeof(int32_t));
  l.items = off;
  off = align256(off + (size_t)l.max_items * sizeof(int4));
  l.seqs = off;
  off = align256(off + (size_t)B * sizeof(int4));
  l.scal = off;
  off = align256(off + (size_t)H * 4 * l.t_pad * sizeof(float));
  l.keybias = off;
  off = align256(off + (size_t)l.t_pad * sizeof(float));
  l.partial = off;
  off = align256(off + T * H * (size_t)(d + 2) * sizeof(float));
  if (d == 64 || d == 128) near_offsets(L, buckets, max_rel, span, l.lt, &l.diag_m0, &l.n_diag);
  const size_t diag_bytes = l.n_diag > 0 ? (size_t)(l.n_diag + 1) * 128 * H * d * 2 : 0;
  l.diag_pk = off;
  off = align256(off + diag_bytes);
  l.diag_pq = off;
  off = align256(off + diag_bytes);
  l.kaug = off;
  off = align256(off + (size_t)l.t_pad * H * 16 * 2);
  l.kaug_sel = off;
  off = align256(off + 256 * 16 * 2);
  l.absel = off;
  off = align256(off + (size_t)H * 16 * 64 * 2);
  l.total = off;
  return l;
}

// Backward sections, after the forward's: row statistics, the two
// bucket-sum tables and the partial position gradients.
struct BwdLayout {
  size_t lse, drow, gc, gp, part, total;
  int splits;
};


int bwd_splits(long long T, int H) {
  long long s = (T + 1023) / 1024;
  s = s < 1 ? 1 : (s > 64 ? 64 : s);
  const long long cap = 65535 / (H > 0 ? H : 1);
  return (int)(s < cap ? s : (cap < 1 ? 1 : cap));
}

BwdLayout make_bwd_layout(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  const Layout f = make_layout(B, H, L, d, buckets, max_rel, span);
  BwdLayout l{};
  const size_t T = (size_t)B * L, R = 2 * (size_t)span;
  size_t off = f.total;
  l.lse = off;
  off = align256(off + T * H * sizeof(float));
  l.drow = off;
  off = align256(off + T * H * sizeof(float));
  l.gc = off;
  off = align256(off + T * H * R * sizeof(float));
  l.gp = off;
  off = align256(off + T * H * R * sizeof(float));
  l.splits = bwd_splits((long long)T, H);
  l.part = off;
  off = align256(off + 2 * (size_t)l.splits * H * R * d * sizeof(float));
  l.total = off;
  return l;
}

// Head size 32 with 16-bit I/O runs the d = 64 tensor-core kernels on
// zero-widened copies: the d = 64 layout first (its header at offset 0), then
// q, k, v, out [T][H][64] and PK, PQ [2 span][H][64].
struct Pad32Layout {
  size_t fwd, q, k, v, o, pk, pq, total;
};

Pad32Layout make_pad32_layout(int B, int H, int L, int buckets, int max_rel, int span) {
  Pad32Layout l{};
  l.fwd = make_layout(B, H, L, 64, buckets, max_rel, span).total;
  const size_t tok = align256((size_t)B * L * H * 64 * 2), pos = align256(2 * (size_t)span * H * 64 * 2);
  l.q = l.fwd;
  l.k = l.q + tok;
  l.v = l.k + tok;
  l.o = l.v + tok;
  l.pk = l.o + tok;
  l.pq = l.pk + pos;
  l.total = l.pq + pos;
  return l;
}

size_t workspace_bytes_for(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  const size_t own = make_layout(B, H, L, d, buckets, max_rel, span).total;
  if (d != 32) return own;
  const size_t wide = make_pad32_layout(B, H, L, buckets, max_rel, span).total;
  return own > wide ? own : wide;
}

// Fast fp32 mode: the fp16 forward's own workspace first (its header, and so
// the device status word, at offset 0), then fp16 copies of q, k, v, out (B L
// rows each), pos_key, pos_query and the conversion's range flag.
struct Fast32Layout {
  size_t inner, q, k, v, o, pk, pq, flag, total;
};

Fast32Layout make_fast32_layout(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  Fast32Layout l{};
  l.inner = workspace_bytes_for(B, H, L, d, buckets, max_rel, span);
  const size_t tok = align256((size_t)B * L * H * d * 2);
  const size_t pos = align256((size_t)2 * span * H * d * 2);
  l.q = align256(l.inner);
  l.k = l.q + tok;
  l.v = l.k + tok;
  l.o = l.v + tok;
  l.pk = l.o + tok;
  l.pq = l.pk + pos;
  l.flag = l.pq + pos;
  l.total = l.flag + 256;
  return l;
}

df_status check_params(int H, int L, int d, df_dtype dtype, int buckets, int max_rel, int span) {
  if (H < 1 || L < 1 || span < 1) return DF_ERR_INVALID_ARG;
  if (dtype != DF_BF16 && dtype != DF_FP16 && dtype != DF_FP32) return DF_ERR_INVALID_ARG;
  if (buckets > 0 && (buckets / 2 < 1 || buckets / 2 >= max_rel - 1)) return DF_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return DF_ERR_UNSUPPORTED;
  if (L > 65536 || span > 65536 || H > 1024) return DF_ERR_UNSUPPORTED;
  return DF_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

df_status build_problem(const void* q, const void* k, const void* v, const void* pk,
                        const void* pq, const uint8_t* key_mask, const int32_t* cu_seqlens,
                        int B, int H, int L, int T, int d, int buckets, int max_rel, int span,
                        df_dtype dtype, void* out, void* ws, size_t ws_bytes, bool need_v,
                        Problem* p) {
  df_status st = check_params(H, L, d, dtype, buckets, max_rel, span);
  if (st != DF_OK) return st;
  if (B < 0 || T < 0) return DF_ERR_INVALID_ARG;
  const bool packed = cu_seqlens != nullptr;
  if ((key_mask == nullptr) == (cu_seqlens == nullptr)) return DF_ERR_INVALID_ARG;
  if ((long long)B * L > (1ll << 26)) return DF_ERR_UNSUPPORTED;
  if (!packed && (long long)T != (long long)B * L) return DF_ERR_INVALID_ARG;
  if (packed && (long long)T > (long long)B * L) return DF_ERR_INVALID_ARG;
  // With no tokens at all the tensors may be empty (NULL data pointers).
  if (T > 0 && (!q || !k || !out || (need_v && !v))) return DF_ERR_INVALID_ARG;
  if (!pk || !pq) return DF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(pk) || !aligned16(pq) || !aligned16(out) ||
      (need_v && !aligned16(v)))
    return DF_ERR_ALIGNMENT;
  const Layout lay = make_layout(B, H, L, d, buckets, max_rel, span);
  if (!ws || ws_bytes < lay.total) return DF_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255) != 0) return DF_ERR_ALIGNMENT;
  char* base = static_cast<char*>(ws);
  Problem& P = *p;
  memset(&P, 0, sizeof(P));
  P.q = q; P.k = k; P.v = v; P.pk = pk; P.pq = pq;
  P.key_mask = key_mask; P.cu_seqlens = cu_seqlens; P.out = out;
  P.B = B; P.H = H; P.L = L; P.T = T; P.d = d;
  P.buckets = buckets; P.max_rel = max_rel; P.span = span;
  P.dtype = (int)dtype; P.packed = packed ? 1 : 0;
  P.kscale = (float)(1.4426950408889634 / sqrt(3.0 * d));
  P.hdr = reinterpret_cast<df_ws_header*>(base + lay.header);
  P.idx = reinterpret_cast<int32_t*>(base + lay.idx);
  P.items = reinterpret_cast<int4*>(base + lay.items);
  P.seqs = reinterpret_cast<int4*>(base + lay.seqs);
  P.scal = reinterpret_cast<float*>(base + lay.scal);
  P.keybias = reinterpret_cast<float*>(base + lay.keybias);
  P.partial = reinterpret_cast<float*>(base + lay.partial);
  P.max_items = lay.max_items;
  P.t_pad = lay.t_pad;
  P.lt = lay.lt;
  P.diag_pk = base + lay.diag_pk;
  P.diag_pq = base + lay.diag_pq;
  P.kaug = base + lay.kaug;
  P.kaug_sel = base + lay.kaug_sel;
  P.absel = base + lay.absel;
  P.n_diag = lay.n_diag;
  P.diag_m0 = lay.diag_m0;
  const unsigned long long wb = g_wait_budget.load();
  P.wait_budget = wb ? wb : kDefaultWaitBudget;
  P.zero_out = 1;
  P.far_possible = far_tiles_possible(L, buckets, max_rel, span, lay.lt, kKBlock) ? 1 : 0;
  // the strict-fp32 kernel and the backward classify 64 x 64 tiles, which reach
  // farther than 128 x 128 ones
  P.scal_needed = far_tiles_possible(L, buckets, max_rel, span, lay.lt, 64) ? 1 : 0;
  return DF_OK;
}

}  // namespace

extern "C" {

const char* df_attn_status_string(df_status s) {
  switch (s) {
    case DF_OK: return "ok";
    case DF_ERR_INVALID_ARG: return "invalid argument";
    case DF_ERR_UNSUPPORTED: return "unsupported configuration";
    case DF_ERR_ALIGNMENT: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case DF_ERR_WORKSPACE: return "workspace missing or too small";
    case DF_ERR_CUDA: return "CUDA runtime error";
    case DF_ERR_DEVICE_TIMEOUT: return "device-side bounded wait ran out";
  }
  return "unknown status";
}

df_status df_attn_supported(int H, int L, int d, df_dtype dtype, int buckets, int max_rel,
                            int span) {
  return check_params(H, L, d, dtype, buckets, max_rel, span);
}

size_t df_attn_workspace_size(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  if (B < 0 || check_params(H, L, d, DF_BF16, buckets, max_rel, span) != DF_OK) return 0;
  return workspace_bytes_for(B, H, L, d, buckets, max_rel, span);
}

df_status df_attn_workspace_layout(int B, int H, int L, int d, int buckets, int max_rel, int span,
                                   df_ws_layout* layout) {
  if (!layout || B < 0) return DF_ERR_INVALID_ARG;
  const df_status st = check_params(H, L, d, DF_BF16, buckets, max_rel, span);
  if (st != DF_OK) return st;
  const Layout l = make_layout(B, H, L, d, buckets, max_rel, span);
  layout->header = l.header;
  layout->idx_table = l.idx;
  layout->items = l.items;
  layout->scalars = l.scal;
  layout->keybias = l.keybias;
  layout->partial = l.partial;
  layout->total = l.total;
  layout->max_items = l.max_items;
  layout->t_pad = l.t_pad;
  layout->table_half = l.lt;
  layout->diag_pk = l.diag_pk;
  layout->diag_pq = l.diag_pq;
  layout->n_diag = l.n_diag;
  layout->diag_m0 = l.diag_m0;
  layout->kaug = l.kaug;
  layout->kaug_sel = l.kaug_sel;
  layout->absel = l.absel;
  return DF_OK;
}

df_status df_attn_plan(const void* q, const void* k, const void* pos_key, const void* pos_query,
                       const uint8_t* key_mask, const int32_t* cu_seqlens, int B, int H, int L,
                       int total_tokens, int d, int buckets, int max_rel, int span,
                       df_dtype dtype, void* out, void* workspace, size_t workspace_bytes,
                       df_stream_t stream) {
  Problem p;
  df_status st = build_problem(q, k, nullptr, pos_key, pos_query, key_mask, cu_seqlens, B, H, L,
                               total_tokens, d, buckets, max_rel, span, dtype, out, workspace,
                               workspace_bytes, false, &p);
  if (st != DF_OK) return st;
  p.scal_needed = 1;  // the planning call always writes every planner output
  return launch_plan(p, (cudaStream_t)stream) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

df_status df_attn_fwd(const void* q, const void* k, const void* v, const void* pos_key,
                      const void* pos_query, const uint8_t* key_mask, const int32_t* cu_seqlens,
                      int B, int H, int L, int total_tokens, int d, int buckets, int max_rel,
                      int span, df_dtype dtype, void* out, void* workspace,
                      size_t workspace_bytes, df_stream_t stream) {
  Problem p;
  df_status st = build_problem(q, k, v, pos_key, pos_query, key_mask, cu_seqlens, B, H, L,
                               total_tokens, d, buckets, max_rel, span, dtype, out, workspace,
                               workspace_bytes, true, &p);
  if (st != DF_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype != DF_FP32 && d == 32 && tc_enabled()) {
    // d = 32 on the tensor cores: widen to 64 with zeros, run the d = 64
    // kernels with the d = 32 scale, narrow the output
    const Pad32Layout pl = make_pad32_layout(B, H, L, buckets, max_rel, span);
    if (workspace_bytes < pl.total) return DF_ERR_WORKSPACE;
    char* base = static_cast<char*>(workspace);
    Problem w;
    st = build_problem(base + pl.q, base + pl.k, base + pl.v, base + pl.pk, base + pl.pq, key_mask,
                       cu_seqlens, B, H, L, total_tokens, 64, buckets, max_rel, span, dtype,
                       base + pl.o, workspace, pl.fwd, true, &w);
    if (st != DF_OK) return st;
    w.kscale = p.kscale;  // the scale of the true head size
    w.scal_in_near = w.far_possible;
    const void* src[5] = {q, k, v, pos_key, pos_query};
    void* dst[5] = {base + pl.q, base + pl.k, base + pl.v, base + pl.pk, base + pl.pq};
    const long long tok_rows = (long long)total_tokens * H, pos_rows = 2ll * span * H;
    const long long rows[5] = {tok_rows, tok_rows, tok_rows, pos_rows, pos_rows};
    if (launch_pad32(src, dst, rows, s) != cudaSuccess || launch_plan(w, s) != cudaSuccess)
      return DF_ERR_CUDA;
    int launches = 0;
    if (launch_tc(w, s, g_prof_start, g_prof_mid, g_prof_stop, &launches) != cudaSuccess) return DF_ERR_CUDA;
    if (launch_unpad32(base + pl.o, out, tok_rows, s) != cudaSuccess) return DF_ERR_CUDA;
    g_last_launches.store(3 + launches);
    return DF_OK;
  }
  // the d = 64 near-tile kernel forms the far tiles' scalars itself
  if (dtype != DF_FP32 && d == 64 && tc_enabled()) p.scal_in_near = p.far_possible;
  if (launch_plan(p, s) != cudaSuccess) return DF_ERR_CUDA;
  int launches = 0;
  cudaError_t e;
  if (dtype != DF_FP32 && d != 32 && tc_enabled()) {
    e = launch_tc(p, s, g_prof_start, g_prof_mid, g_prof_stop, &launches);
  } else {
    if (g_prof_start) cudaEventRecord(g_prof_start, s);
    if (g_prof_mid) cudaEventRecord(g_prof_mid, s);
    e = launch_simt(p, s, &launches);
    if (g_prof_stop) cudaEventRecord(g_prof_stop, s);
  }
  if (e != cudaSuccess) return DF_ERR_CUDA;
  g_last_launches.store(1 + launches);
  return DF_OK;
}

size_t df_attn_fwd_fp32_fast_workspace_size(int B, int H, int L, int d, int buckets, int max_rel,
                                            int span) {
  if (B < 0 || check_params(H, L, d, DF_FP16, buckets, max_rel, span) != DF_OK) return 0;
  return make_fast32_layout(B, H, L, d, buckets, max_rel, span).total;
}

df_status df_attn_fwd_fp32_fast(const void* q, const void* k, const void* v, const void* pos_key,
                                const void* pos_query, const uint8_t* key_mask,
                                const int32_t* cu_seqlens, int B, int H, int L, int total_tokens,
                                int d, int buckets, int max_rel, int span, void* out,
                                void* workspace, size_t workspace_bytes, df_stream_t stream) {
  df_status st = check_params(H, L, d, DF_FP16, buckets, max_rel, span);
  if (st != DF_OK) return st;
  if (B < 0 || total_tokens < 0 || (long long)total_tokens > (long long)B * L) return DF_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !out)) return DF_ERR_INVALID_ARG;
  if (!pos_key || !pos_query) return DF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(pos_key) || !aligned16(pos_query) ||
      !aligned16(out))
    return DF_ERR_ALIGNMENT;
  const Fast32Layout fl = make_fast32_layout(B, H, L, d, buckets, max_rel, span);
  if (!workspace || workspace_bytes < fl.total) return DF_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255) != 0) return DF_ERR_ALIGNMENT;
  char* base = static_cast<char*>(workspace);
  // every remaining check of the fp16 forward, before anything is enqueued
  Problem chk;
  st = build_problem(base + fl.q, base + fl.k, base + fl.v, base + fl.pk, base + fl.pq, key_mask,
                     cu_seqlens, B, H, L, total_tokens, d, buckets, max_rel, span, DF_FP16,
                     base + fl.o, workspace, fl.inner, true, &chk);
  if (st != DF_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int* flag = reinterpret_cast<int*>(base + fl.flag);
  const long long tok = (long long)total_tokens * H * d, pos = 2ll * span * H * d;
  const float* src[5] = {static_cast<const float*>(q), static_cast<const float*>(k),
                         static_cast<const float*>(v), static_cast<const float*>(pos_key),
                         static_cast<const float*>(pos_query)};
  void* dst[5] = {base + fl.q, base + fl.k, base + fl.v, base + fl.pk, base + fl.pq};
  const long long n[5] = {tok, tok, tok, pos, pos};
  if (launch_to_half(src, dst, n, flag, s) != cudaSuccess) return DF_ERR_CUDA;
  st = df_attn_fwd(base + fl.q, base + fl.k, base + fl.v, base + fl.pk, base + fl.pq, key_mask,
                   cu_seqlens, B, H, L, total_tokens, d, buckets, max_rel, span, DF_FP16,
                   base + fl.o, workspace, fl.inner, stream);
  if (st != DF_OK) return st;
  const int inner = g_last_launches.load();
  if (launch_to_float(base + fl.o, static_cast<float*>(out), tok, flag, workspace, s) != cudaSuccess)
    return DF_ERR_CUDA;
  g_last_launches.store(inner + 2);
  return DF_OK;
}

size_t df_attn_bwd_workspace_size(int B, int H, int L, int d, int buckets, int max_rel, int span) {
  if (B < 0 || check_params(H, L, d, DF_BF16, buckets, max_rel, span) != DF_OK) return 0;
  return make_bwd_layout(B, H, L, d, buckets, max_rel, span).total;
}

df_status df_attn_bwd(const void* q, const void* k, const void* v, const void* pos_key,
                      const void* pos_query, const void* dout, const uint8_t* key_mask,
                      const int32_t* cu_seqlens, int B, int H, int L, int total_tokens, int d,
                      int buckets, int max_rel, int span, df_dtype dtype, float* dq, float* dk,
                      float* dv, float* dpos_key, float* dpos_query, void* workspace,
                      size_t workspace_bytes, df_stream_t stream) {
  BwdProblem b;
  memset(&b, 0, sizeof(b));
  df_status st = build_problem(q, k, v, pos_key, pos_query, key_mask, cu_seqlens, B, H, L,
                               total_tokens, d, buckets, max_rel, span, dtype, dq, workspace,
                               workspace_bytes, true, &b.f);
  if (st != DF_OK) return st;
  const int T = total_tokens;
  if (!dpos_key || !dpos_query || (T > 0 && (!dout || !dk || !dv))) return DF_ERR_INVALID_ARG;
  if (!aligned16(dpos_key) || !aligned16(dpos_query) ||
      (T > 0 && (!aligned16(dout) || !aligned16(dk) || !aligned16(dv))))
    return DF_ERR_ALIGNMENT;
  const BwdLayout bl = make_bwd_layout(B, H, L, d, buckets, max_rel, span);
  if (workspace_bytes < bl.total) return DF_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  b.f.zero_out = 0;  // `out` is dq here: the planner must leave it alone
  b.dout = dout;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  b.dpk = dpos_key;
  b.dpq = dpos_query;
  b.lse = reinterpret_cast<float*>(base + bl.lse);
  b.drow = reinterpret_cast<float*>(base + bl.drow);
  b.gc = reinterpret_cast<float*>(base + bl.gc);
  b.gp = reinterpret_cast<float*>(base + bl.gp);
  b.part = reinterpret_cast<float*>(base + bl.part);
  b.R = 2 * span;
  b.splits = bwd_splits(T, H);
  b.kchunk = T > 0 ? (T + b.splits - 1) / b.splits : 1;
  b.sscale = (float)(1.0 / sqrt(3.0 * d));
  cudaStream_t s = (cudaStream_t)stream;
  const size_t R = (size_t)b.R;
  // rows outside every sequence (and masked ones) must read as zero
  if (T > 0) {
    const size_t grad = (size_t)T * H * d * sizeof(float), gsum = (size_t)T * H * R * sizeof(float);
    if (cudaMemsetAsync(dq, 0, grad, s) != cudaSuccess || cudaMemsetAsync(dk, 0, grad, s) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, grad, s) != cudaSuccess || cudaMemsetAsync(b.gc, 0, gsum, s) != cudaSuccess ||
        cudaMemsetAsync(b.gp, 0, gsum, s) != cudaSuccess)
      return DF_ERR_CUDA;
  } else {
    const size_t pos = R * H * d * sizeof(float);
    if (cudaMemsetAsync(dpos_key, 0, pos, s) != cudaSuccess ||
        cudaMemsetAsync(dpos_query, 0, pos, s) != cudaSuccess)
      return DF_ERR_CUDA;
  }
  if (launch_plan(b.f, s) != cudaSuccess) return DF_ERR_CUDA;
  int launches = 0;
  if (launch_bwd(b, s, g_prof_start, g_prof_mid, g_prof_stop, &launches) != cudaSuccess)
    return DF_ERR_CUDA;
  g_last_launches.store(1 + launches);
  return DF_OK;
}

df_status df_attn_get_device_status(void* workspace, df_stream_t stream) {
  if (!workspace) return DF_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DF_ERR_CUDA;
  df_ws_header h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DF_ERR_CUDA;
  const int32_t zero[2] = {0, 0};
  if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return DF_ERR_CUDA;
  return (df_status)h.status;
}

df_status df_rel_index_table(int buckets, int max_rel, int span, int max_len, int32_t* idx,
                             df_stream_t stream) {
  if (!idx || max_len < 1 || max_len > 65536 || span < 1) return DF_ERR_INVALID_ARG;
  if (buckets > 0 && (buckets / 2 < 1 || buckets / 2 >= max_rel - 1)) return DF_ERR_INVALID_ARG;
  if (((uintptr_t)idx & 3) != 0) return DF_ERR_ALIGNMENT;
  return launch_index_table(buckets, max_rel, span, max_len, idx, (cudaStream_t)stream) ==
                 cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

void df_attn_set_profile_events(df_event_t start, df_event_t stop) {
  g_prof_start = (cudaEvent_t)start;
  g_prof_stop = (cudaEvent_t)stop;
}

void df_attn_set_profile_split(df_event_t mid) { g_prof_mid = (cudaEvent_t)mid; }

void df_attn_set_wait_budget(unsigned long long cycles) { g_wait_budget.store(cycles); }

int df_attn_last_launch_count(void) { return g_last_launches.load(); }

}  // extern "C"
