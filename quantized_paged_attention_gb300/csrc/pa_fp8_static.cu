// pa_decode_fp8_static: the fp8 decode step for callers that cannot allocate
// device memory. The partition partials, which pa_decode_fp8 keeps in a
// caller-supplied workspace, live here in one file-scope device array that
// every GPU loading the library holds until the process exits.
#include <mutex>

#include "qpa.h"
#include "common.cuh"
#include "qpa_internal.h"

// The shared scratch. Host code sees only a host-side stand-in under this
// name; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char qpa_fp8_static_scratch[QPA_FP8_STATIC_SCRATCH_BYTES];

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (no
// link-time dependency on the driver library); null if unavailable.
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// One looked-up address per (device, context): the symbol's device address is
// only valid in the context it was looked up in.
struct Entry {
  int dev;
  CUcontext ctx;
  void* ptr;
};
constexpr int kMaxEntries = 64;
std::mutex g_mu;
Entry g_entries[kMaxEntries];
int g_num_entries = 0;

// Device address of the scratch array in the current device's current
// context. The first call in a (device, context) looks it up, with that device
// current, and caches it.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (ctx)
    for (int i = 0; i < g_num_entries; ++i)
      if (g_entries[i].dev == dev && g_entries[i].ctx == ctx) return g_entries[i].ptr;
  // not looked up in this context yet (or no context is current, which the
  // lookup itself makes the device's primary one)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, qpa_fp8_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
  if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return nullptr;
  Entry e{dev, ctx, p};
  if (g_num_entries < kMaxEntries) g_entries[g_num_entries++] = e;
  else g_entries[dev % kMaxEntries] = e;      // table full: reuse a slot (looked up again when evicted)
  return p;
}
}  // namespace

extern "C" int pa_decode_fp8_static(const void* q, const uint8_t* kv_cache, const int32_t* block_table,
                                    const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                                    int num_partitions, void* out, const qpa_fp8_desc* d, void* stream) {
  const size_t need = pa_decode_fp8_workspace_size(d, num_partitions);
  if (need == 0)   // invalid arguments or nothing to do: let the regular entry point report which
    return pa_decode_fp8(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, out, d,
                         nullptr, 0, stream);
  if (need > QPA_FP8_STATIC_SCRATCH_BYTES) return QPA_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return QPA_ERR_CUDA;
  return pa_decode_fp8(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions, out, d, ws,
                       QPA_FP8_STATIC_SCRATCH_BYTES, stream);
}
