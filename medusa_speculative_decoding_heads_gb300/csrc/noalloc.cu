// medusa_tree_attention_noalloc: tree attention whose scratch memory is a
// library-owned static device array, for callers that cannot allocate.
//
// Who needs this: a serving engine that reserves almost all device memory for
// its KV cache at start-up and forbids later cudaMalloc calls, code that runs
// inside a host framework whose caching allocator owns every device byte, or a
// plug-in that is handed only the tensors it works on. Such callers can pass
// their inputs and outputs but cannot provide the workspace that
// medusa_tree_attention wants for its split-KV partial results.
//
// The array below holds those partials instead. It is fixed at build time
// (MEDUSA_NOALLOC_SCRATCH_BYTES), so every GPU that loads the library keeps it
// resident until the process exits. All calls share it: two calls whose
// kernels overlap on the GPU (different streams, or graphs replayed
// concurrently) race on it. Each call writes every partial it later reads, so
// nothing has to be cleared between calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace medusa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MEDUSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static array on the current device. The host-side
// symbol is only a stand-in, so the address is looked up once per device (with
// that device current) and cached.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_tree_attention_noalloc(const medusa_cfg* cfg, const void* Q, const void* Kc, const void* Vc,
                                             const int32_t* L, const uint64_t* anc_bits, void* O,
                                             medusa_stream_t stream) {
  int s = check_cfg_public(cfg);
  if (s != MEDUSA_OK) return s;
  if (!Q || !Kc || !Vc || !L || !anc_bits || !O) return MEDUSA_ERR_INVALID_ARG;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Kc) |
                         reinterpret_cast<uintptr_t>(Vc) | reinterpret_cast<uintptr_t>(O)) & 15u;
  if (mis) return MEDUSA_ERR_INVALID_ARG;
  if (attention_workspace(*cfg) > (size_t)MEDUSA_NOALLOC_SCRATCH_BYTES) return MEDUSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MEDUSA_ERR_CUDA;
  return launch_attention(*cfg, Q, Kc, Vc, L, anc_bits, O, scratch, (cudaStream_t)stream) == cudaSuccess
             ? MEDUSA_OK
             : MEDUSA_ERR_CUDA;
}
