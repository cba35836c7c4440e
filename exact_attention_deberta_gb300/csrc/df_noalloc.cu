// df_attn_fwd_noalloc: the fused forward for callers that cannot allocate device
// memory.
//
// df_attn_fwd needs a caller-provided workspace.  Some callers have no way to
// get one: a plug-in running inside a host application that owns every byte of
// device memory and exposes no allocator to it, or a latency-critical service
// that forbids cudaMalloc / cudaFree (and the device-wide synchronisation they
// can cause) once it has started.  This entry point serves them: its scratch is
// a fixed array in the library's own device image, so the call itself allocates
// nothing.  The caller still provides the inputs and the output.
//
// The array holds DF_ATTN_NOALLOC_SCRATCH_BYTES on every GPU that loads the
// library, for as long as the process lives.  Its device address is looked up
// on every call with the caller's device current, so a reset of the device
// (which reloads the module) never leaves a stale address behind.
//
// Errors the kernels raise on the device (a bounded wait that ran out, bad
// cu_seqlens) land in the status word at the start of the shared array;
// df_attn_noalloc_get_device_status reads and clears it.
#include "df_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DF_ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on
// every call (cheap once the module is loaded), so that no address outlives a
// reset of the device's primary context.  The host-side name g_noalloc_scratch
// is only a stand-in for the symbol and must never reach a kernel;
// cudaGetSymbolAddress turns it into the device address.
df_status scratch_on_current_device(void** addr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DF_ERR_CUDA;
  *addr = p;
  return DF_OK;
}

}  // namespace

extern "C" df_status df_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                         const void* pos_key, const void* pos_query,
                                         const uint8_t* key_mask, const int32_t* cu_seqlens,
                                         int B, int H, int L, int total_tokens, int d,
                                         int buckets, int max_rel, int span, df_dtype dtype,
                                         void* out, df_stream_t stream) {
  const size_t need = df_attn_workspace_size(B, H, L, d, buckets, max_rel, span);
  if (need > (size_t)DF_ATTN_NOALLOC_SCRATCH_BYTES) return DF_ERR_WORKSPACE;
  void* scratch = nullptr;
  const df_status st = scratch_on_current_device(&scratch);
  if (st != DF_OK) return st;
  // Every section of the scratch is written by the planning kernel before it is
  // read (including the status word), so nothing has to be cleared here.
  return df_attn_fwd(q, k, v, pos_key, pos_query, key_mask, cu_seqlens, B, H, L, total_tokens, d,
                     buckets, max_rel, span, dtype, out, scratch,
                     (size_t)DF_ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" df_status df_attn_noalloc_get_device_status(df_stream_t stream) {
  void* scratch = nullptr;
  const df_status st = scratch_on_current_device(&scratch);
  if (st != DF_OK) return st;
  return df_attn_get_device_status(scratch, stream);
}
