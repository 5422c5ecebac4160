// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at the moment they need a decode step:
// code running inside a custom allocator or memory-pool callback, runtimes that have
// reserved all device memory up front and hand out no scratch, or plug-ins that are
// given only their input and output buffers.  For them nsa_sparse_decode_noalloc runs
// the same decode kernels as nsa_sparse_decode, with the scratch taken from a
// fixed-size array in device memory that this library owns.  That array is a
// file-scope __device__ object: every GPU that loads the library holds it until the
// process exits.
#include <cuda.h>

#include <mutex>

#include "nsa.h"
#include "launch.h"

using namespace nsa;

namespace {

// 16 MiB: a decode step of 32 sequences x 32768 tokens, 16 heads, 2 kv-heads, d = 128,
// top-k 64 needs about 3.3 MB of scratch; at that shape up to 310 sequences fit.
constexpr size_t kScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // CUDA context the address belongs to (0: unknown)
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context, or 0 when there is none or it
// cannot be read.  A device reset or a context torn down and created again gets a new id
// (and a new copy of the scratch array), so a cached address is only reused within the
// context it was looked up in.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    looked_up = true;
  }
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device.  Host code cannot use the
// array's name as a device pointer: the address is asked of the runtime once per device
// and context (the first call on a device does this set-up; make that first call before
// any stream capture), and asked again whenever the current context has changed.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchAddr& s = g_scratch[dev];
  const unsigned long long id = current_context_id();
  if (!s.ptr || id == 0 || id != s.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // also makes the device's context current
    if (e != cudaSuccess) return e;
    s.ptr = p;
    s.ctx_id = current_context_id();
  }
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" NSA_API size_t nsa_sparse_decode_noalloc_max_bytes(void) { return kScratchBytes; }

extern "C" NSA_API nsa_status nsa_sparse_decode_noalloc(int batch, const int32_t* seqlens, int max_len, int h,
                                                      int h_kv, int d, const void* q, const void* k_cache,
                                                      const void* v_cache, const void* k_cmp_cache, int kernel,
                                                      int stride, int block_size, int n_init, int n_local, int k,
                                                      float scale, int32_t* idx_out, void* o,
                                                      cudaStream_t stream) {
  // sizes the decode step does not support get the regular entry point's message
  if (nsa_status st = decode_check_sizes(batch, max_len, h, h_kv, d, kernel, stride, block_size, n_init, n_local, k))
    return st;
  if (batch == 0) return NSA_OK;
  const size_t need = nsa_sparse_decode_workspace_size(batch, max_len, h, h_kv, d, kernel, stride, block_size, k);
  if (need > kScratchBytes) {
    set_error("nsa_sparse_decode_noalloc: this step needs %zu bytes of scratch, more than the fixed %zu bytes; "
              "use nsa_sparse_decode with a caller-provided workspace",
              need, kScratchBytes);
    return NSA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    set_error("nsa_sparse_decode_noalloc: cannot resolve the scratch array: %s", cudaGetErrorString(e));
    return NSA_ERR_CUDA;
  }
  // every other check (pointers, alignment, memory kinds) is the regular entry point's
  return nsa_sparse_decode(batch, seqlens, max_len, h, h_kv, d, q, k_cache, v_cache, k_cmp_cache, kernel, stride,
                           block_size, n_init, n_local, k, scale, idx_out, o, scratch, kScratchBytes, stream);
}
