// Fixed device scratch for mla_decode_no_alloc.
//
// Some callers cannot allocate device memory when they decode: a serving
// engine whose caching allocator already owns nearly all of HBM (a cudaMalloc
// outside that pool fails or fragments it), or a host thread that must not
// stall on the device-wide synchronisation cudaMalloc and cudaFree can imply.
// For them the split-KV partials, the copied work list and the device error
// word live in one array that is part of this library's device image: every
// GPU that loads the library holds kNoAllocScratchBytes here until the
// process exits, whether or not the entry point is ever called.
//
// The array's name, used in host code, is only a host-side stand-in for the
// symbol, not a device address. The device address is looked up once per
// device with that device current (cudaGetSymbolAddress) and cached; that is
// the pointer the kernels get.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace mla {
namespace {

static_assert(kNoAllocScratchBytes == MLA_NO_ALLOC_SCRATCH_BYTES,
              "scratch size in the header and the library differ");

static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

cudaError_t no_alloc_scratch(int device, uint8_t** ptr) {
  *ptr = nullptr;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    // `device` is the current device: the caller has just read it back.
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[device] = static_cast<uint8_t*>(p);
  }
  *ptr = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace mla
