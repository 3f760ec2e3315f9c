// moda_bwd_noalloc: the backward without a caller-provided workspace.
//
// moda_bwd needs T*Hq floats of scratch (the per-row dot products of dO and o)
// and takes them from the caller. Some callers cannot hand over device memory
// for it: code whose device memory belongs to another allocator (a
// framework's caching allocator, a fixed pool sized up front) and that must
// not take memory from outside it, and code that must not risk cudaMalloc's
// implicit device synchronisation on a latency-critical path. For them this
// entry point runs the same kernels on a fixed scratch array compiled into the
// library, so neither side allocates.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its 4 MiB until the process exits. In host code the name
// g_bwd_scratch is only a host-side stand-in for the symbol, never a device
// address; its device address is looked up with cudaGetSymbolAddress (with
// that device current) on the first call on each device, and again whenever
// the device's current context is not the one it was looked up in (after a
// cudaDeviceReset the module's variables live in a new context).
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "moda.h"
#include "moda_internal.h"

namespace {

constexpr int64_t kScratchFloats = int64_t{1} << 20;  // rows T*Hq the array holds
static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchEntry {
  void* ctx = nullptr;
  float* addr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];

}  // namespace

extern "C" moda_status moda_bwd_noalloc(const void* q, const void* k, const void* v,
                                        const void* kd, const void* vd, const void* o,
                                        const float* lse, const void* dO, int T, int Hq, int Hk,
                                        int d, int L, float scale, float* dq, float* dk, float* dv,
                                        float* dkd, float* dvd, moda_stream_t stream) {
  if ((int64_t)T * Hq > kScratchFloats)
    return moda::report(MODA_ERR_UNSUPPORTED,
                        "T*Hq = %lld rows exceed the fixed scratch of %lld rows; use moda_bwd "
                        "with a caller workspace",
                        (long long)T * Hq, (long long)kScratchFloats);
  // the device must be one the library runs on before its symbols are touched
  int dev = -1;
  moda_status st = moda::checked_device(&dev);
  if (st != MODA_OK) return st;
  if (dev >= kMaxDevices)
    return moda::report(MODA_ERR_NO_DEVICE, "device ordinal %d; libmoda serves devices 0..%d",
                        dev, kMaxDevices - 1);
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ScratchEntry& ent = g_scratch[dev];
    void* ctx = moda::current_context();
    if (!ent.addr || !ctx || ctx != ent.ctx) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p)
        return moda::report(MODA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                            cudaGetErrorString(e));
      ent.addr = static_cast<float*>(p);
      ent.ctx = moda::current_context();
    }
    scratch = ent.addr;
  }
  // Every element of the scratch that the kernels read is first written by
  // the same call (the delta kernel fills all T*Hq rows), so nothing needs
  // clearing between calls.
  return moda_bwd(q, k, v, kd, vd, o, lse, dO, T, Hq, Hk, d, L, scale, dq, dk, dv, dkd, dvd,
                  scratch, stream);
}
