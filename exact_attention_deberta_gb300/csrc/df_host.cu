// Host-buffer forward: the copies to and from the device overlap the fused
// kernels.
//
// Sequences (padded: batch rows) are independent problems (DisentangledFlash
// 0.2.0 README, "Packed unpadded inference": each sequence of a packed batch
// attends only within itself), so a batch can be cut into groups of whole
// sequences and each group run as its own df_attn_fwd call with identical
// results.  Three streams form a pipeline over two device slots:
//
//   copy-in stream      group g's q, k, v (and mask rows) host -> slot g % 2
//   compute stream g%2  df_attn_fwd(group g) from slot g % 2, with the slot's
//                       own workspace
//   copy-out stream     slot g % 2's output -> host
//
// so the copy-in of group g + 1 and the copy-out of group g - 1 run while
// group g computes, and the kernels of group g + 1 can start on the SMs that
// group g's last work items leave idle.  A slot is refilled only after the
// forward that read it has finished, and its output is overwritten only after
// the copy-out that read it has finished (events).  Everything starts after
// the work already on the caller's stream, which waits for the last copy-out
// before the call returns, so synchronising that stream completes everything.
// The streams and events are created once per device and reused; a mutex
// serialises the enqueueing of concurrent calls.
#include "df_common.cuh"

#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

namespace {

struct Pipe {
  int device = -1;
  cudaStream_t in = nullptr, out = nullptr;
  cudaStream_t comp[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr;
  cudaEvent_t loaded[2] = {nullptr, nullptr};    // slot inputs on the device
  cudaEvent_t computed[2] = {nullptr, nullptr};  // forward of the slot done
  cudaEvent_t drained[2] = {nullptr, nullptr};   // slot output copied out
};

std::mutex g_mu;
// One set of streams and events per device, created on the device's first
// call and kept for the process (calls on several devices each use their own).
constexpr int kMaxDevices = 64;
Pipe g_pipes[kMaxDevices];

void destroy_pipe(Pipe& p) {
  cudaStream_t* ss[] = {&p.in, &p.out, &p.comp[0], &p.comp[1]};
  for (cudaStream_t* st : ss)
    if (*st) cudaStreamDestroy(*st);
  cudaEvent_t* evs[] = {&p.start, &p.loaded[0], &p.loaded[1], &p.computed[0], &p.computed[1],
                        &p.drained[0], &p.drained[1]};
  for (cudaEvent_t* e : evs)
    if (*e) cudaEventDestroy(*e);
  p = Pipe{};
}

// The current device's pipe, or nullptr.  A pipe is published (device set)
// only once every stream and event of it exists; a partial one is destroyed.
Pipe* pipe_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  Pipe& slot = g_pipes[dev];
  if (slot.device == dev) return &slot;
  Pipe p;
  bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaStreamCreateWithFlags(&p.comp[i], cudaStreamNonBlocking) == cudaSuccess;
  cudaEvent_t* evs[] = {&p.start, &p.loaded[0], &p.loaded[1], &p.computed[0], &p.computed[1],
                        &p.drained[0], &p.drained[1]};
  for (cudaEvent_t* e : evs)
    if (ok) ok = cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    destroy_pipe(p);
    return nullptr;
  }
  p.device = dev;
  slot = p;
  return &slot;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct HostLayout {
  size_t ws[2], ws_bytes, pk, pq, cu, slot[2], q, k, v, o, mask, total;
  long long cap_tokens;  // tokens one slot holds
  int cap_rows;          // padded: batch rows one slot holds
};

long long group_capacity(int B, int L, long long group_tokens) {
  const long long auto_cap = ((long long)B * L + 3) / 4;
  const long long want = group_tokens > 0 ? group_tokens : auto_cap;
  return std::max<long long>(want, L);
}

HostLayout host_layout(int B, int H, int L, int d, int buckets, int max_rel, int span, size_t es,
                       long long group_tokens) {
  HostLayout l{};
  l.cap_tokens = group_capacity(B, L, group_tokens);
  l.cap_rows = (int)std::max<long long>(1, l.cap_tokens / L);
  const size_t row = (size_t)H * d * es;
  size_t off = 0;
  l.ws_bytes = df_attn_workspace_size(B, H, L, d, buckets, max_rel, span);
  for (int i = 0; i < 2; ++i) {  // one forward workspace per slot, the first at offset 0
    l.ws[i] = off;
    off = align256(off + l.ws_bytes);
  }
  l.pk = off;
  off = align256(off + 2 * (size_t)span * row);
  l.pq = off;
  off = align256(off + 2 * (size_t)span * row);
  l.cu = off;  // every group's rebased cu_seqlens: at most 2 B + 1 entries
  off = align256(off + (2 * (size_t)B + 2) * sizeof(int32_t));
  const size_t tensor = align256((size_t)l.cap_tokens * row);
  l.q = 0;
  l.k = tensor;
  l.v = 2 * tensor;
  l.o = 3 * tensor;
  l.mask = 4 * tensor;
  const size_t slot = align256(4 * tensor + (size_t)l.cap_rows * L);
  l.slot[0] = off;
  l.slot[1] = off + slot;
  l.total = off + 2 * slot;
  return l;
}

size_t dtype_size(df_dtype t) { return t == DF_FP32 ? 4 : 2; }

}  // namespace

extern "C" size_t df_attn_fwd_host_scratch_size(int B, int H, int L, int d, int buckets, int max_rel,
                                                int span, df_dtype dtype, long long group_tokens) {
  if (B < 1 || df_attn_supported(H, L, d, dtype, buckets, max_rel, span) != DF_OK || group_tokens < 0)
    return 0;
  return host_layout(B, H, L, d, buckets, max_rel, span, dtype_size(dtype), group_tokens).total;
}

extern "C" df_status df_attn_fwd_host(const void* q, const void* k, const void* v, const void* pos_key,
                                      const void* pos_query, const uint8_t* key_mask,
                                      const int32_t* cu_seqlens, int B, int H, int L, int total_tokens,
                                      int d, int buckets, int max_rel, int span, df_dtype dtype, void* out,
                                      long long group_tokens, void* scratch, size_t scratch_bytes,
                                      df_stream_t stream) {
  // ---- host-side checks (no CUDA call before they pass)
  df_status st = df_attn_supported(H, L, d, dtype, buckets, max_rel, span);
  if (st != DF_OK) return st;
  if (B < 1 || total_tokens < 0 || group_tokens < 0) return DF_ERR_INVALID_ARG;
  if ((key_mask == nullptr) == (cu_seqlens == nullptr)) return DF_ERR_INVALID_ARG;
  if (!pos_key || !pos_query) return DF_ERR_INVALID_ARG;
  const bool packed = cu_seqlens != nullptr;
  if (!packed && (long long)total_tokens != (long long)B * L) return DF_ERR_INVALID_ARG;
  if (packed) {  // host memory: the whole contract can be checked here
    if (cu_seqlens[0] != 0 || cu_seqlens[B] != total_tokens) return DF_ERR_INVALID_ARG;
    for (int s = 0; s < B; ++s) {
      const int n = cu_seqlens[s + 1] - cu_seqlens[s];
      if (n < 0 || n > L) return DF_ERR_INVALID_ARG;
    }
  }
  if (total_tokens > 0 && (!q || !k || !v || !out)) return DF_ERR_INVALID_ARG;
  const size_t es = dtype_size(dtype);
  const HostLayout lay = host_layout(B, H, L, d, buckets, max_rel, span, es, group_tokens);
  if (!scratch || scratch_bytes < lay.total) return DF_ERR_WORKSPACE;
  if (((uintptr_t)scratch & 255) != 0) return DF_ERR_ALIGNMENT;

  // ---- groups of whole sequences (padded: of batch rows)
  struct Group {
    int s0, s1;          // sequences (rows) [s0, s1)
    long long t0, t1;    // tokens [t0, t1)
    int cu_off;          // rebased cu_seqlens of the group inside the cu section
  };
  // The first groups ramp up from L tokens (one full sequence), doubling, to
  // the slot capacity: the pipeline starts computing after a short copy-in.
  std::vector<Group> groups;
  std::vector<int32_t> cu_all;
  auto ramp = [&](size_t gi) {
    return gi >= 40 ? lay.cap_tokens : std::min<long long>(lay.cap_tokens, (long long)L << gi);
  };
  if (packed) {
    int s = 0;
    while (s < B) {
      const long long cap = ramp(groups.size());
      Group g{s, s, cu_seqlens[s], cu_seqlens[s], (int)cu_all.size()};
      while (g.s1 < B && (g.s1 == g.s0 || cu_seqlens[g.s1 + 1] - g.t0 <= cap)) ++g.s1;
      g.t1 = cu_seqlens[g.s1];
      for (int e = g.s0; e <= g.s1; ++e) cu_all.push_back(cu_seqlens[e] - (int32_t)g.t0);
      groups.push_back(g);
      s = g.s1;
    }
  } else {
    for (int r = 0; r < B;) {
      const int rows = (int)std::max<long long>(1, ramp(groups.size()) / L);
      const int r1 = std::min(B, r + rows);
      groups.push_back(Group{r, r1, (long long)r * L, (long long)r1 * L, 0});
      r = r1;
    }
  }

  std::lock_guard<std::mutex> lock(g_mu);
  Pipe* pp = pipe_for_current_device();
  if (!pp) return DF_ERR_CUDA;
  Pipe& P = *pp;
  cudaStream_t cs = (cudaStream_t)stream;
  char* base = static_cast<char*>(scratch);
  const size_t row = (size_t)H * d * es;
  const size_t pos_bytes = 2 * (size_t)span * row;
  bool ok = cudaEventRecord(P.start, cs) == cudaSuccess &&
            cudaStreamWaitEvent(P.in, P.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(P.out, P.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(P.comp[0], P.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(P.comp[1], P.start, 0) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(base + lay.pk, pos_key, pos_bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(base + lay.pq, pos_query, pos_bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
  if (packed && ok)
    ok = cudaMemcpyAsync(base + lay.cu, cu_all.data(), cu_all.size() * sizeof(int32_t),
                         cudaMemcpyHostToDevice, P.in) == cudaSuccess;
  if (!ok) return DF_ERR_CUDA;
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  char* ho = static_cast<char*>(out);
  for (size_t gi = 0; gi < groups.size(); ++gi) {
    const Group& g = groups[gi];
    const int sl = (int)(gi & 1);
    char* slot = base + lay.slot[sl];
    const size_t off = (size_t)g.t0 * row, bytes = (size_t)(g.t1 - g.t0) * row;
    // copy in, once the forward that last read this slot is done
    if (gi >= 2) ok = ok && cudaStreamWaitEvent(P.in, P.computed[sl], 0) == cudaSuccess;
    if (bytes) {
      ok = ok && cudaMemcpyAsync(slot + lay.q, hq + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
      ok = ok && cudaMemcpyAsync(slot + lay.k, hk + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
      ok = ok && cudaMemcpyAsync(slot + lay.v, hv + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
    }
    if (!packed)
      ok = ok && cudaMemcpyAsync(slot + lay.mask, key_mask + (size_t)g.s0 * L, (size_t)(g.s1 - g.s0) * L,
                                 cudaMemcpyHostToDevice, P.in) == cudaSuccess;
    ok = ok && cudaEventRecord(P.loaded[sl], P.in) == cudaSuccess;
    // the forward, once the inputs landed and the previous output left the slot
    cudaStream_t comp = P.comp[sl];
    ok = ok && cudaStreamWaitEvent(comp, P.loaded[sl], 0) == cudaSuccess;
    if (gi >= 2) ok = ok && cudaStreamWaitEvent(comp, P.drained[sl], 0) == cudaSuccess;
    if (!ok) return DF_ERR_CUDA;
    const int Bg = g.s1 - g.s0;
    const int Tg = (int)(g.t1 - g.t0);
    st = df_attn_fwd(slot + lay.q, slot + lay.k, slot + lay.v, base + lay.pk, base + lay.pq,
                     packed ? nullptr : reinterpret_cast<const uint8_t*>(slot + lay.mask),
                     packed ? reinterpret_cast<const int32_t*>(base + lay.cu) + g.cu_off : nullptr, Bg, H, L,
                     Tg, d, buckets, max_rel, span, dtype, slot + lay.o, base + lay.ws[sl], lay.ws_bytes,
                     (df_stream_t)comp);
    if (st != DF_OK) return st;
    ok = cudaEventRecord(P.computed[sl], comp) == cudaSuccess;
    // copy out
    ok = ok && cudaStreamWaitEvent(P.out, P.computed[sl], 0) == cudaSuccess;
    if (bytes)
      ok = ok && cudaMemcpyAsync(ho + off, slot + lay.o, bytes, cudaMemcpyDeviceToHost, P.out) == cudaSuccess;
    ok = ok && cudaEventRecord(P.drained[sl], P.out) == cudaSuccess;
    if (!ok) return DF_ERR_CUDA;
  }
  // the caller's stream completes with the last copy-out of both slots
  for (size_t sl = 0; sl < std::min<size_t>(2, groups.size()); ++sl)
    if (cudaStreamWaitEvent(cs, P.drained[sl], 0) != cudaSuccess) return DF_ERR_CUDA;
  return DF_OK;
}
