// cp_decode_attention_noalloc: the fused decode (partials + merge in one launch) for callers
// that cannot hand the library device memory when they call it.  Its scratch is a fixed array
// built into this translation unit, so only processes that load this unit's module (the first
// call of this entry point does) hold it, one copy per GPU, until they exit.
//
// Host code must never use the array's host-side name as a device pointer: the device address
// is looked up with cudaGetSymbolAddress, once per CUDA context (with the device current), and
// passed to the decode launcher.  The cache is keyed by the driver's context id, which is never
// reused, so a context that was torn down and recreated (cudaDeviceReset, a destroyed primary
// context) gets its address looked up afresh instead of a stale one.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

static __device__ __align__(256) unsigned char g_decode_scratch[CP_NOALLOC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

void* driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return ptr;
}

// Id of the calling thread's current context (0 if none or unknown).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
  static CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kSlots = 64;
struct Slot {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_mu;
Slot g_slots[kSlots] = {};
int g_next = 0;

// Device address of the scratch array in the current context.  The first call in a context
// resolves it (loading this unit's module and its array on that GPU); later calls reuse it.
cudaError_t scratch_address(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);  // the device the address must belong to is current
  if (e != cudaSuccess) return e;
  unsigned long long id = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0) {
    for (int i = 0; i < kSlots; ++i)
      if (g_slots[i].ctx_id == id && g_slots[i].addr != nullptr) {
        *ptr = g_slots[i].addr;
        return cudaSuccess;
      }
  }
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_decode_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_ctx_id();  // the lookup above may have created the context
  if (id != 0) {
    g_slots[g_next] = Slot{id, addr};
    g_next = (g_next + 1) % kSlots;
  }
  *ptr = addr;
  return cudaSuccess;
}

}  // namespace

extern "C" cp_status cp_decode_attention_noalloc(const cp_decode_args* a, void* out,
                                                 float* out_lse, void* stream) {
  const cp_status st = cp_check_decode_args_for_fused(a, out);
  if (st != CP_OK) return st;
  size_t ol = 0, oo = 0;
  const size_t need = cp_decode_ws_layout(a->num_seqs, a->num_q_heads, a->num_kv_heads,
                                          a->head_dim, a->cp * a->num_splits, &ol, &oo);
  if (need > CP_NOALLOC_SCRATCH_BYTES)
    return cp_fail_detail(CP_ERR_INVALID_ARG,
                          "cp_decode_attention_noalloc needs %zu bytes of scratch but its static "
                          "array holds %zu: use fewer splits or a smaller batch",
                          need, (size_t)CP_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) return cp_launch_status(e, "static scratch address");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero whatever an earlier call left behind
  e = cudaMemsetAsync(ws, 0, ol, s);
  if (e != cudaSuccess) return cp_launch_status(e, "static scratch clear");
  CpDecodeWorkspace w;
  w.counters = static_cast<int32_t*>(ws);
  w.partial_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + ol);
  w.partial_out = reinterpret_cast<float*>(static_cast<char*>(ws) + oo);
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  return cp_launch_status(cp_launch_decode_fused(*a, scale, w, out, out_lse, s),
                          "fused decode (static scratch) launch");
}
