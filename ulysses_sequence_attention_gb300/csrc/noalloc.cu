// noalloc.cu — the backward pass for callers that cannot allocate device memory.
//
// ulysses_attn_bwd takes its workspace from the caller. Callers inside a host
// runtime that owns the GPU's memory (a plugin given only its buffers, a
// server that must not allocate after start-up, a framework allocator that
// tracks every byte) have no way to provide one. This file holds a fixed
// workspace in the library itself and runs the unchanged backward on it.
#include <mutex>

#include "internal.cuh"

namespace {

// The workspace of ulysses_attn_bwd_noalloc: the backward's fp32 row planes
// (-LSE*log2(e) and D). It lives for the lifetime of the process on every
// device that loads the library. Calls share it; each backward writes the
// rows before it reads them.
static __device__ __align__(256) unsigned char g_bwd_scratch[ULYSSES_NOALLOC_SCRATCH_BYTES];

// Device address of g_bwd_scratch for each device. In host code the symbol is
// only a host-side stand-in, so the address comes from cudaGetSymbolAddress,
// with that device current. The lookup also loads this file's module on the
// device (modules load lazily), and with it the array: ulysses_create does it
// during set-up (noalloc_setup), so that the first ulysses_attn_bwd_noalloc
// finds the array in place and commits no memory. Every create looks the
// address up again: a handle made after a cudaDeviceReset (which destroys
// the handles made before it) so sees the array of the new context.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int lookup(int dev) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
    cudaGetLastError();  // leave no sticky error for the caller's next check
    return ULYSSES_ERR_CUDA;
  }
  g_scratch_addr[dev] = p;
  return ULYSSES_OK;
}

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ULYSSES_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ULYSSES_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    const int st = lookup(dev);
    if (st != ULYSSES_OK) return st;
  }
  *out = g_scratch_addr[dev];
  return ULYSSES_OK;
}

}  // namespace

namespace uly {
// Set-up of the no-alloc scratch on the current device (from ulysses_create).
// A failure here is not the handle's: the no-alloc call tries once more and
// reports it.
void noalloc_setup() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  lookup(dev);
}
}  // namespace uly

extern "C" int ulysses_attn_bwd_noalloc(ulysses_t h, const void* const* q, const void* const* k,
                                        const void* const* v, const void* const* o, const void* const* dO,
                                        const float* const* lse, void* const* dq, void* const* dk,
                                        void* const* dv, void* stream) {
  if (!h) return ULYSSES_ERR_INVALID_ARG;
  // The row planes only: dQ is recomputed here even when the handle's dS
  // budget would store dS.
  const size_t need = uly::workspace_bytes(*reinterpret_cast<const uly::Layer*>(h), false);
  if (need > (size_t)ULYSSES_NOALLOC_SCRATCH_BYTES) return ULYSSES_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != ULYSSES_OK) return st;
  return uly::attn_bwd_entry(h, q, k, v, o, dO, lse, dq, dk, dv, scratch, stream, false);
}
