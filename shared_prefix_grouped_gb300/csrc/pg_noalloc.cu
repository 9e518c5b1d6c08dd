// Grouped-attention forward that allocates nothing: its scratch (the RoPE-rotated Q and K the
// attention kernel reads) lives in one file-scope device array instead of a caller workspace.
//
// The array is a module-scope __device__ object: every GPU that loads this library holds it until
// the process exits.  Host code may not pass the array's name to a kernel (on the host that name
// is only a stand-in for the device object), so its device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "pg_internal.h"

namespace pg {

namespace {

static __device__ __align__(256) unsigned char g_fwd_scratch[PG_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

pg_status scratch_address(void** out) {
  int dev = 0;
  pg_status st = cuda_check(cudaGetDevice(&dev), "pg_grouped_attn_fwd_noalloc: cudaGetDevice");
  if (st != PG_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("pg_grouped_attn_fwd_noalloc: device index %d out of range", dev);
    return PG_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_fwd_scratch),
                    "pg_grouped_attn_fwd_noalloc: cudaGetSymbolAddress");
    if (st != PG_OK) return st;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return PG_OK;
}

}  // namespace

}  // namespace pg

using namespace pg;

extern "C" pg_status pg_grouped_attn_fwd_noalloc(const pg_layout* layout, pg_dtype dtype,
                                                 int32_t heads_q, int32_t heads_kv,
                                                 int32_t head_dim, const void* q, const void* k,
                                                 const void* v, void* o, float* lse,
                                                 const pg_opts* opts, pg_stream_t stream) {
  size_t need = 0;
  pg_status st = pg_workspace_size(layout, dtype, heads_q, heads_kv, head_dim, opts, 0, &need);
  if (st != PG_OK) return st;
  if (need > (size_t)PG_NOALLOC_SCRATCH_BYTES) {
    set_error("pg_grouped_attn_fwd_noalloc: this problem needs %zu bytes of scratch, more than "
              "the built-in %llu; use pg_grouped_attn_fwd with a caller workspace",
              need, (unsigned long long)PG_NOALLOC_SCRATCH_BYTES);
    return PG_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != PG_OK) return st;
  // Nothing in the scratch has to start at zero: every byte the call reads (rotated Q and K) is
  // written by the same call before it is read.
  return pg_grouped_attn_fwd(layout, dtype, heads_q, heads_kv, head_dim, q, k, v, o, lse, opts,
                             scratch, (size_t)PG_NOALLOC_SCRATCH_BYTES, stream);
}
