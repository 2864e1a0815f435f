// grs_grad_norm_sq_noalloc: the global squared gradient norm computed from
// the accumulator with scratch memory that the library owns statically, for
// callers that cannot allocate device memory.
//
// Who cannot allocate: a process whose framework caching allocator has
// already reserved (nearly) all of the device's memory, where a fresh
// cudaMalloc fails or fragments the pool; latency-critical code that cannot
// afford the implicit device synchronisation cudaMalloc/cudaFree may incur;
// and hosts that only receive device pointers from another runtime and have
// no allocator of their own.  They pass the accumulator and the output; the
// scratch (per-tile partial sums, second-level sums, a ticket counter) is a
// file-scope array in device memory.
//
// The array is GRS_NOALLOC_SCRATCH_BYTES (4 MiB) on every GPU that loads
// the library, held until the process exits.  All calls share it and it
// keeps the last call's contents; the ticket counter is cleared on the
// stream before each launch.  Calls that overlap on the GPU (two streams,
// or two host threads) race on the array and must be serialised by the
// caller.  The first call on a device resolves the array's device address
// (cudaGetSymbolAddress) with that device current; make that first call
// before any stream capture.  The address is cached for the process: a
// cudaDeviceReset unloads the module with the context, after which the
// cached address is stale (documented as unsupported in grs.h).
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = GRS_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

grs_status fail(grs_status s, const std::string& msg) {
  grs::set_last_error(msg);
  return s;
}

}  // namespace

extern "C" grs_status grs_grad_norm_sq_noalloc(const grs_plan* p, const float* acc, int32_t n_micro,
                                               double* d_norm_sq, void* stream) {
  if (p == nullptr || acc == nullptr || d_norm_sq == nullptr)
    return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq_noalloc: NULL argument");
  if (p->device < 0)
    return fail(GRS_ERR_NO_DEVICE, "grs_grad_norm_sq_noalloc: plan was created with GRS_PLAN_HOST_ONLY");
  if (n_micro < 1) return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq_noalloc: n_micro must be >= 1");
  if ((reinterpret_cast<uintptr_t>(acc) & 15u) != 0 || (reinterpret_cast<uintptr_t>(d_norm_sq) & 7u) != 0)
    return fail(GRS_ERR_ALIGNMENT, "grs_grad_norm_sq_noalloc: misaligned pointer");
  const int64_t need = grs::ws_bytes(p->n_red_tiles);
  if (need > static_cast<int64_t>(kScratchBytes))
    return fail(GRS_ERR_SHAPE, "grs_grad_norm_sq_noalloc: the plan needs " + std::to_string(need) +
                                   " bytes of scratch (" + std::to_string(p->n_red_tiles) +
                                   " reduction tiles); the static array holds " +
                                   std::to_string(kScratchBytes) + " bytes");
  if (p->device >= kMaxDevices)
    return fail(GRS_ERR_INVALID_ARG, "grs_grad_norm_sq_noalloc: device index beyond the supported range");
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess)
    return fail(GRS_ERR_CUDA, "grs_grad_norm_sq_noalloc: cudaGetDevice failed");
  if (prev != p->device && cudaSetDevice(p->device) != cudaSuccess)
    return fail(GRS_ERR_CUDA, "grs_grad_norm_sq_noalloc: cannot select the plan's device");
  grs_status st = GRS_OK;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[p->device] == nullptr) {
      // One-time set-up on this device (the plan's device is current).
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) {
        st = fail(GRS_ERR_CUDA, std::string("grs_grad_norm_sq_noalloc: cudaGetSymbolAddress: ") +
                                    cudaGetErrorString(e));
      } else {
        g_scratch_ptr[p->device] = ptr;
      }
    }
    scratch = g_scratch_ptr[p->device];
  }
  if (st == GRS_OK) {
    uint8_t* ws = static_cast<uint8_t*>(scratch);
    cudaError_t e = cudaMemsetAsync(ws + grs::ws_ticket_offset(p->n_red_tiles), 0, sizeof(unsigned int),
                                    static_cast<cudaStream_t>(stream));
    int le = 0;
    if (e == cudaSuccess) le = grs::launch_norm(p, acc, n_micro, ws, 0, d_norm_sq, stream);
    if (e != cudaSuccess || le != 0) {
      const cudaError_t ee = e != cudaSuccess ? e : static_cast<cudaError_t>(le);
      st = fail(GRS_ERR_CUDA, std::string("grs_grad_norm_sq_noalloc: ") + cudaGetErrorName(ee) + " (" +
                                  cudaGetErrorString(ee) + ")");
    }
  }
  if (prev != p->device) cudaSetDevice(prev);
  return st;
}
