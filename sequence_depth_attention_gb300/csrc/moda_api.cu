// C-ABI entry points of libmoda.so (declared in include/moda.h): argument
// validation, the per-device kernel error word, and dispatch to the kernels.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "moda.h"
#include "moda_internal.h"

// Latched by kernels whose bounded waits give up; read and cleared by
// moda_get_device_error. One copy per device (module-scope device variable).
__device__ unsigned int g_moda_err = 0;

// Tile queues of the persistent forward: {next tile, CTAs finished} per
// slot. A launch takes the next slot in turn; its last CTA puts both back to
// zero, so a slot is clean again when the launch has finished.
constexpr int kQueueSlots = 64;
__device__ unsigned int g_moda_queue[kQueueSlots][2] = {};

namespace {

thread_local char g_detail[256] = "";

moda_status fail(moda_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moda_status fail(moda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return s;
}

moda_status ok() {
  g_detail[0] = '\0';
  return MODA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
struct DeviceEntry {
  void* ctx = nullptr;            // context the cached addresses belong to
  unsigned int* err = nullptr;    // device address of g_moda_err in it
  unsigned int* queue = nullptr;  // device address of g_moda_queue in it
  int sms = 0;
};
std::atomic<unsigned int> g_queue_seq{0};
DeviceEntry g_dev[kMaxDevices];

// Current device, its error-word address and SM count; checks that it is
// an sm_103 part (the only target the library is compiled for). The address
// is cached per device together with the context it was resolved in, and
// resolved again when the current context differs (after cudaDeviceReset the
// runtime creates a new primary context, and the module's variables move).
moda_status device_state(int* dev_out, unsigned int** err_out, int* sms_out,
                         unsigned int** queue_out = nullptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0)
    return fail(MODA_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= kMaxDevices)
    return fail(MODA_ERR_NO_DEVICE, "device ordinal %d; libmoda serves devices 0..%d", dev,
                kMaxDevices - 1);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceEntry& ent = g_dev[dev];
  void* ctx = moda::current_context();
  if (!ent.err || !ctx || ctx != ent.ctx) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
      return fail(MODA_ERR_NO_DEVICE, "device %d is sm_%d%d; libmoda is built for sm_103a", dev,
                  major, minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moda_err);
    if (e != cudaSuccess || !p)
      return fail(MODA_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
    ent.err = (unsigned int*)p;
    void* qp = nullptr;
    e = cudaGetSymbolAddress(&qp, g_moda_queue);
    if (e != cudaSuccess || !qp)
      return fail(MODA_ERR_CUDA, "cudaGetSymbolAddress(tile queues): %s", cudaGetErrorString(e));
    ent.queue = (unsigned int*)qp;
    ent.sms = sms;
    ent.ctx = moda::current_context();  // bound by now
  }
  *dev_out = dev;
  *err_out = ent.err;
  *sms_out = ent.sms;
  if (queue_out) *queue_out = ent.queue + 2 * (g_queue_seq.fetch_add(1) % kQueueSlots);
  return MODA_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

namespace moda {
void* current_context() {
  static PFN_cuCtxGetCurrent_v4000 get = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  }();
  CUcontext c = nullptr;
  if (!get || get(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

moda_status checked_device(int* dev) {
  unsigned int* err;
  int sms;
  return device_state(dev, &err, &sms);
}

moda_status report(moda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return s;
}
}  // namespace moda

extern "C" {

const char* moda_status_string(moda_status s) {
  switch (s) {
    case MODA_OK: return "MODA_OK";
    case MODA_ERR_INVALID_ARG: return "MODA_ERR_INVALID_ARG";
    case MODA_ERR_UNSUPPORTED: return "MODA_ERR_UNSUPPORTED";
    case MODA_ERR_MISALIGNED: return "MODA_ERR_MISALIGNED";
    case MODA_ERR_CUDA: return "MODA_ERR_CUDA";
    case MODA_ERR_TIMEOUT: return "MODA_ERR_TIMEOUT";
    case MODA_ERR_NO_DEVICE: return "MODA_ERR_NO_DEVICE";
  }
  return "MODA_ERR_UNKNOWN";
}

const char* moda_last_error_detail(void) { return g_detail; }

// The address a kernel must use for p: p itself for device or managed memory,
// the device mapping for page-locked host memory; nullptr (and the reason)
// for memory the device cannot address, such as pageable host memory.
static const void* device_view(const void* p, bool allow_host, const char** why) {
  cudaPointerAttributes at;
  const cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    *why = "the runtime does not know this address";
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeHost && allow_host) {
    if (at.devicePointer) return at.devicePointer;
    *why = "page-locked host memory without a device mapping";
    return nullptr;
  }
  *why = at.type == cudaMemoryTypeHost ? "host memory where device memory is required"
                                       : "pageable host memory (page-lock it, or copy it to the device)";
  return nullptr;
}

moda_status moda_pack_depth(const void* src, void* dst, int L, int T, int Hk, int d,
                            moda_stream_t stream) {
  if (L < 0) return fail(MODA_ERR_INVALID_ARG, "L = %d < 0", L);
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (Hk < 1) return fail(MODA_ERR_INVALID_ARG, "Hk = %d < 1", Hk);
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (L == 0) return ok();
  if (!src || !dst) return fail(MODA_ERR_INVALID_ARG, "NULL src or dst with L = %d", L);
  if (!aligned16(src) || !aligned16(dst))
    return fail(MODA_ERR_MISALIGNED, "src or dst not 16-byte aligned");
  const size_t bytes = (size_t)L * T * Hk * d * 2;
  if (overlaps(src, bytes, dst, bytes)) return fail(MODA_ERR_INVALID_ARG, "src and dst overlap");
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  const char* why = "";
  const void* ksrc = device_view(src, true, &why);
  if (!ksrc) return fail(MODA_ERR_INVALID_ARG, "src: %s", why);
  if (!device_view(dst, false, &why)) return fail(MODA_ERR_INVALID_ARG, "dst: %s", why);
  cudaError_t e = moda::launch_pack_depth(ksrc, dst, L, T, Hk, d, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "pack_depth launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_depth_write(const void* src, void* dst, int T, int Hk, int d, int L, int slot,
                             moda_stream_t stream) {
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (Hk < 1) return fail(MODA_ERR_INVALID_ARG, "Hk = %d < 1", Hk);
  if (L < 1) return fail(MODA_ERR_INVALID_ARG, "L = %d < 1", L);
  if (slot < 0 || slot >= L) return fail(MODA_ERR_INVALID_ARG, "slot = %d outside [0, %d)", slot, L);
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  if (!src || !dst) return fail(MODA_ERR_INVALID_ARG, "NULL src or dst");
  if (!aligned16(src) || !aligned16(dst))
    return fail(MODA_ERR_MISALIGNED, "src or dst not 16-byte aligned");
  if (overlaps(src, (size_t)T * Hk * d * 2, dst, (size_t)Hk * T * L * d * 2))
    return fail(MODA_ERR_INVALID_ARG, "src and dst overlap");
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_depth_write(src, dst, T, Hk, d, L, slot, nullptr, err, sms,
                                           (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "depth_write launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_depth_write_at(const void* src, void* dst, int T, int Hk, int d, int L,
                                const int* slot, moda_stream_t stream) {
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (Hk < 1) return fail(MODA_ERR_INVALID_ARG, "Hk = %d < 1", Hk);
  if (L < 1) return fail(MODA_ERR_INVALID_ARG, "L = %d < 1", L);
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  if (!src || !dst || !slot) return fail(MODA_ERR_INVALID_ARG, "NULL src, dst or slot");
  if (!aligned16(src) || !aligned16(dst))
    return fail(MODA_ERR_MISALIGNED, "src or dst not 16-byte aligned");
  if (((uintptr_t)slot & 3u) != 0) return fail(MODA_ERR_MISALIGNED, "slot not 4-byte aligned");
  if (overlaps(src, (size_t)T * Hk * d * 2, dst, (size_t)Hk * T * L * d * 2))
    return fail(MODA_ERR_INVALID_ARG, "src and dst overlap");
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_depth_write(src, dst, T, Hk, d, L, 0, slot, err, sms,
                                           (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "depth_write launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t moda_depth_mass_workspace_bytes(int T, int Hk, int L) {
  if (T < 1 || Hk < 1 || L < 1) return 0;
  return moda::depth_mass_workspace_floats(T, Hk, L) * sizeof(float);
}

moda_status moda_depth_mass(const void* q, const void* kd, const float* lse, int T, int Hq,
                            int Hk, int d, int L, float scale, float* mass, float* workspace,
                            size_t workspace_bytes, moda_stream_t stream) {
  if (!q || !kd || !lse || !mass || !workspace)
    return fail(MODA_ERR_INVALID_ARG, "NULL input, output or workspace pointer");
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (L < 1) return fail(MODA_ERR_INVALID_ARG, "L = %d < 1", L);
  if (Hk < 1 || Hq < 1) return fail(MODA_ERR_INVALID_ARG, "Hq = %d, Hk = %d", Hq, Hk);
  if (Hq % Hk != 0) return fail(MODA_ERR_INVALID_ARG, "Hq = %d not a multiple of Hk = %d", Hq, Hk);
  if (!(scale > 0.f) || scale == __builtin_inff())
    return fail(MODA_ERR_INVALID_ARG, "scale must be positive and finite");
  const int G = Hq / Hk;
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(MODA_ERR_UNSUPPORTED, "G = Hq/Hk = %d (supported: 1, 2, 4, 8, 16)", G);
  if (T > (1 << 24)) return fail(MODA_ERR_UNSUPPORTED, "T = %d > 2^24", T);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  const size_t need = moda::depth_mass_workspace_floats(T, Hk, L) * sizeof(float);
  if (workspace_bytes < need)
    return fail(MODA_ERR_INVALID_ARG, "workspace of %zu bytes; %zu needed", workspace_bytes, need);
  if (!aligned16(q) || !aligned16(kd) || !aligned16(lse) || !aligned16(mass) || !aligned16(workspace))
    return fail(MODA_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  const size_t mb = (size_t)Hk * L * 4;
  const void* ins[3] = {q, kd, lse};
  const size_t insz[3] = {(size_t)T * Hq * d * 2, (size_t)Hk * T * L * d * 2, (size_t)T * Hq * 4};
  for (int i = 0; i < 3; ++i)
    if (overlaps(mass, mb, ins[i], insz[i]) || overlaps(workspace, need, ins[i], insz[i]))
      return fail(MODA_ERR_INVALID_ARG, "the output or the workspace overlaps an input");
  if (overlaps(mass, mb, workspace, need))
    return fail(MODA_ERR_INVALID_ARG, "mass and workspace overlap");
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  moda::DepthMassArgs a{q, kd, lse, T, Hq, Hk, d, L, G, scale, mass, workspace};
  cudaError_t e = moda::launch_depth_mass(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "depth_mass launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_depth_cache_admit(int* slot_age, const float* mass, int Hk, int S, int recent,
                                   int new_age, int* slot, moda_stream_t stream) {
  if (!slot_age || !mass || !slot) return fail(MODA_ERR_INVALID_ARG, "NULL pointer");
  if (S < 1) return fail(MODA_ERR_INVALID_ARG, "S = %d < 1", S);
  if (Hk < 1) return fail(MODA_ERR_INVALID_ARG, "Hk = %d < 1", Hk);
  if (recent < 0) return fail(MODA_ERR_INVALID_ARG, "recent = %d < 0", recent);
  if (new_age < 0) return fail(MODA_ERR_INVALID_ARG, "new_age = %d < 0", new_age);
  if (S > 1024) return fail(MODA_ERR_UNSUPPORTED, "S = %d > 1024", S);
  if (((uintptr_t)slot_age & 3u) || ((uintptr_t)mass & 3u) || ((uintptr_t)slot & 3u))
    return fail(MODA_ERR_MISALIGNED, "a pointer is not 4-byte aligned");
  if (overlaps(slot_age, (size_t)S * 4, slot, 4) || overlaps(mass, (size_t)Hk * S * 4, slot, 4) ||
      overlaps(slot_age, (size_t)S * 4, mass, (size_t)Hk * S * 4))
    return fail(MODA_ERR_INVALID_ARG, "slot_age, mass and slot must not overlap");
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_cache_admit(slot_age, mass, Hk, S, recent, new_age, slot,
                                           (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "cache_admit launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_kv_proj_write(const void* x, const void* wk, const void* wv, int T, int Dm,
                               int Hk, int d, int L, int slot, void* kd, void* vd,
                               moda_stream_t stream) {
  if (!x || !wk || !wv || !kd || !vd) return fail(MODA_ERR_INVALID_ARG, "NULL input or output");
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (Hk < 1) return fail(MODA_ERR_INVALID_ARG, "Hk = %d < 1", Hk);
  if (Dm < 1) return fail(MODA_ERR_INVALID_ARG, "Dm = %d < 1", Dm);
  if (L < 1) return fail(MODA_ERR_INVALID_ARG, "L = %d < 1", L);
  if (slot < 0 || slot >= L) return fail(MODA_ERR_INVALID_ARG, "slot = %d outside [0, %d)", slot, L);
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (Dm % 64 != 0) return fail(MODA_ERR_UNSUPPORTED, "Dm = %d is not a multiple of 64", Dm);
  if (T > (1 << 24)) return fail(MODA_ERR_UNSUPPORTED, "T = %d > 2^24", T);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  if ((int64_t)Hk * d > (1 << 24))
    return fail(MODA_ERR_UNSUPPORTED, "Hk*d = %lld output features exceed 2^24", (long long)Hk * d);
  const void* all[] = {x, wk, wv, kd, vd};
  for (const void* p : all)
    if (!aligned16(p)) return fail(MODA_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  const size_t xb = (size_t)T * Dm * 2, wb = (size_t)Hk * d * Dm * 2;
  const size_t db = (size_t)Hk * T * L * d * 2;
  const void* ins[] = {x, wk, wv};
  const size_t insz[] = {xb, wb, wb};
  for (int b = 0; b < 3; ++b)
    if (overlaps(kd, db, ins[b], insz[b]) || overlaps(vd, db, ins[b], insz[b]))
      return fail(MODA_ERR_INVALID_ARG, "an output overlaps an input");
  if (overlaps(kd, db, vd, db)) return fail(MODA_ERR_INVALID_ARG, "kd and vd overlap");
  moda::KvProjArgs a{};
  a.x = x; a.wk = wk; a.wv = wv;
  a.T = T; a.Dm = Dm; a.Hk = Hk; a.d = d; a.L = L; a.slot = slot;
  a.kd = kd; a.vd = vd;
  int dev;
  moda_status st = device_state(&dev, &a.err, &a.num_sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_kv_proj(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "kv_proj launch: %s", cudaGetErrorString(e));
  return ok();
}

// Validation shared by the forward entry points; fills *out on success.
// The forward's shape and scale rules (everything but the pointers).
static moda_status check_fwd_shape(int T, int Hq, int Hk, int d, int L, float scale) {
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (L < 0) return fail(MODA_ERR_INVALID_ARG, "L = %d < 0", L);
  if (Hk < 1 || Hq < 1) return fail(MODA_ERR_INVALID_ARG, "Hq = %d, Hk = %d", Hq, Hk);
  if (Hq % Hk != 0) return fail(MODA_ERR_INVALID_ARG, "Hq = %d not a multiple of Hk = %d", Hq, Hk);
  if (!(scale > 0.f) || scale == __builtin_inff())
    return fail(MODA_ERR_INVALID_ARG, "scale must be positive and finite");
  const int G = Hq / Hk;
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(MODA_ERR_UNSUPPORTED, "G = Hq/Hk = %d (supported: 1, 2, 4, 8, 16)", G);
  if (T > (1 << 24)) return fail(MODA_ERR_UNSUPPORTED, "T = %d > 2^24", T);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  // the kernels address packed depth rows with 32-bit coordinates, and a
  // tile's depth blocks may reach up to 128*L rows past its last own row
  if ((int64_t)Hk * T * L + 128LL * L > 0x7fffffffLL)
    return fail(MODA_ERR_UNSUPPORTED, "Hk*T*L = %lld packed depth rows exceed 2^31 - 1 - 128*L",
                (long long)Hk * T * L);
  return MODA_OK;
}

static moda_status prepare_fwd(const void* q, const void* k, const void* v, const void* kd,
                               const void* vd, int T, int Hq, int Hk, int d, int L, float scale,
                               void* o, float* lse, moda::FwdArgs* out, int layer_major = 0) {
  if (!q || !k || !v || !o) return fail(MODA_ERR_INVALID_ARG, "NULL q, k, v or o");
  if (L > 0 && (!kd || !vd)) return fail(MODA_ERR_INVALID_ARG, "NULL kd or vd with L = %d", L);
  moda_status sst = check_fwd_shape(T, Hq, Hk, d, L, scale);
  if (sst != MODA_OK) return sst;
  const int G = Hq / Hk;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (L > 0 && (!aligned16(kd) || !aligned16(vd))) || (lse && !aligned16(lse)))
    return fail(MODA_ERR_MISALIGNED, "a tensor pointer is not 16-byte aligned");
  const size_t qb = (size_t)T * Hq * d * 2, kvb = (size_t)T * Hk * d * 2;
  const size_t db = (size_t)Hk * T * L * d * 2, lb = lse ? (size_t)T * Hq * 4 : 0;
  const void* ins[5] = {q, k, v, L ? kd : nullptr, L ? vd : nullptr};
  const size_t insz[5] = {qb, kvb, kvb, db, db};
  for (int i = 0; i < 5; ++i) {
    if (overlaps(o, qb, ins[i], insz[i]) || overlaps(lse, lb, ins[i], insz[i]))
      return fail(MODA_ERR_INVALID_ARG, "an output overlaps an input");
  }
  if (overlaps(o, qb, lse, lb)) return fail(MODA_ERR_INVALID_ARG, "o and lse overlap");

  moda::FwdArgs& a = *out;
  a = moda::FwdArgs{};
  a.q = q; a.k = k; a.v = v;
  a.kd = L ? kd : nullptr; a.vd = L ? vd : nullptr;
  a.T = T; a.Hq = Hq; a.Hk = Hk; a.d = d; a.L = L; a.G = G;
  a.scale = scale; a.o = o; a.lse = lse;
  a.layer_major = layer_major;
  return device_state(&a.device, &a.err, &a.num_sms, &a.queue);
}

moda_status moda_fwd(const void* q, const void* k, const void* v, const void* kd,
                     const void* vd, int T, int Hq, int Hk, int d, int L, float scale, void* o,
                     float* lse, moda_stream_t stream) {
  moda::FwdArgs a;
  moda_status st = prepare_fwd(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, &a);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_fwd_tc(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "moda_fwd launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_fwd_layer_major(const void* q, const void* k, const void* v, const void* kd,
                                 const void* vd, int T, int Hq, int Hk, int d, int L, float scale,
                                 void* o, float* lse, moda_stream_t stream) {
  moda::FwdArgs a;
  moda_status st = prepare_fwd(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, &a, 1);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_fwd_tc(a, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(MODA_ERR_CUDA, "moda_fwd_layer_major launch: %s", cudaGetErrorString(e));
  return ok();
}

// Device workspace of moda_fwd_layer_major_host: the inputs, o and lse, each
// region starting on a 256-byte boundary.
namespace {
struct HostFwdLayout {
  size_t q, k, v, kd, vd, o, lse, total;
};

bool host_fwd_layout(int T, int Hq, int Hk, int d, int L, HostFwdLayout* h) {
  if (T < 1 || Hq < 1 || Hk < 1 || d < 1 || L < 0) return false;
  // reject sizes whose byte counts would not fit in 62 bits
  const double big = (double)T * (double)(Hq > Hk ? Hq : Hk) * (double)d * (double)(L > 1 ? L : 1);
  if (big > 4.0e17) return false;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t qb = (size_t)T * Hq * d * 2, kvb = (size_t)T * Hk * d * 2;
  const size_t db = (size_t)L * T * Hk * d * 2, lb = (size_t)T * Hq * 4;
  size_t off = 0;
  h->q = off; off += up(qb);
  h->k = off; off += up(kvb);
  h->v = off; off += up(kvb);
  h->kd = off; off += up(db);
  h->vd = off; off += up(db);
  h->o = off; off += up(qb);
  h->lse = off; off += up(lb);
  h->total = off;
  return true;
}
}  // namespace

size_t moda_fwd_host_workspace_bytes(int T, int Hq, int Hk, int d, int L) {
  HostFwdLayout h;
  return host_fwd_layout(T, Hq, Hk, d, L, &h) ? h.total : 0;
}

moda_status moda_fwd_layer_major_host(const void* q, const void* k, const void* v, const void* kd,
                                      const void* vd, int T, int Hq, int Hk, int d, int L,
                                      float scale, void* o, float* lse, void* workspace,
                                      size_t workspace_bytes, moda_stream_t stream) {
  if (!workspace) return fail(MODA_ERR_INVALID_ARG, "NULL workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MODA_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  moda_status st = check_fwd_shape(T, Hq, Hk, d, L, scale);
  if (st != MODA_OK) return st;
  HostFwdLayout h;
  if (!host_fwd_layout(T, Hq, Hk, d, L, &h)) return fail(MODA_ERR_UNSUPPORTED, "tensor sizes overflow");
  if (!q || !k || !v || !o) return fail(MODA_ERR_INVALID_ARG, "NULL host q, k, v or o");
  if (L > 0 && (!kd || !vd)) return fail(MODA_ERR_INVALID_ARG, "NULL host kd or vd with L = %d", L);
  if (workspace_bytes < h.total)
    return fail(MODA_ERR_INVALID_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes, h.total);
  const size_t qb = (size_t)T * Hq * d * 2, kvb = (size_t)T * Hk * d * 2;
  const size_t db = (size_t)L * T * Hk * d * 2, lb = lse ? (size_t)T * Hq * 4 : 0;
  if (overlaps(o, qb, lse, lb)) return fail(MODA_ERR_INVALID_ARG, "o and lse overlap");
  const void* host[7] = {q, k, v, L ? kd : nullptr, L ? vd : nullptr, o, lse};
  const size_t hostsz[7] = {qb, kvb, kvb, db, db, qb, lb};
  for (int i = 0; i < 7; ++i)
    if (overlaps(host[i], hostsz[i], workspace, h.total))
      return fail(MODA_ERR_INVALID_ARG, "a host buffer overlaps the workspace");
  // the device copies' placement in the workspace, and the device
  moda::FwdArgs a;
  st = prepare_fwd(ws + h.q, ws + h.k, ws + h.v, L ? ws + h.kd : nullptr,
                               L ? ws + h.vd : nullptr, T, Hq, Hk, d, L, scale, ws + h.o,
                               lse ? reinterpret_cast<float*>(ws + h.lse) : nullptr, &a, 1);
  if (st != MODA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t dst[5] = {h.q, h.k, h.v, h.kd, h.vd};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 5 && e == cudaSuccess; ++i)
    if (hostsz[i]) e = cudaMemcpyAsync(ws + dst[i], host[i], hostsz[i], cudaMemcpyDefault, s);
  if (e != cudaSuccess)
    return fail(MODA_ERR_CUDA, "moda_fwd_layer_major_host input copy: %s", cudaGetErrorString(e));
  e = moda::launch_fwd_tc(a, s);
  if (e != cudaSuccess)
    return fail(MODA_ERR_CUDA, "moda_fwd_layer_major_host launch: %s", cudaGetErrorString(e));
  e = cudaMemcpyAsync(o, ws + h.o, qb, cudaMemcpyDefault, s);
  if (e == cudaSuccess && lse) e = cudaMemcpyAsync(lse, ws + h.lse, lb, cudaMemcpyDefault, s);
  if (e != cudaSuccess)
    return fail(MODA_ERR_CUDA, "moda_fwd_layer_major_host output copy: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_fwd_depth_cc(const void* q, const void* k, const void* v, const void* kd,
                              const void* vd, int T, int Hq, int Hk, int d, int L, float scale,
                              void* o, float* lse, moda_stream_t stream) {
  if (!lse) return fail(MODA_ERR_INVALID_ARG, "lse is required (it carries the merge state)");
  moda::FwdArgs a;
  moda_status st = prepare_fwd(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, &a);
  if (st != MODA_OK) return st;
  // pass 1: the sequence part alone (the forward with L = 0)
  moda::FwdArgs seq = a;
  seq.L = 0;
  seq.kd = seq.vd = nullptr;
  cudaError_t e = moda::launch_fwd_tc(seq, (cudaStream_t)stream);
  // pass 2: the depth slots on CUDA cores, merged into o and lse
  if (e == cudaSuccess && a.L > 0) e = moda::launch_fwd_depth_cc(a, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(MODA_ERR_CUDA, "moda_fwd_depth_cc launch: %s", cudaGetErrorString(e));
  return ok();
}

static moda_status bwd_impl(const void* q, const void* k, const void* v, const void* kd,
                            const void* vd, const void* o, const float* lse, const void* dO, int T,
                            int Hq, int Hk, int d, int L, float scale, float* dq, float* dk,
                            float* dv, float* dkd, float* dvd, float* delta, moda_stream_t stream,
                            int layer_major) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !delta)
    return fail(MODA_ERR_INVALID_ARG, "NULL input, output or workspace pointer");
  if (T < 1) return fail(MODA_ERR_INVALID_ARG, "T = %d < 1", T);
  if (L < 0) return fail(MODA_ERR_INVALID_ARG, "L = %d < 0", L);
  if (Hk < 1 || Hq < 1) return fail(MODA_ERR_INVALID_ARG, "Hq = %d, Hk = %d", Hq, Hk);
  if (Hq % Hk != 0) return fail(MODA_ERR_INVALID_ARG, "Hq = %d not a multiple of Hk = %d", Hq, Hk);
  if (L > 0 && (!kd || !vd || !dkd || !dvd))
    return fail(MODA_ERR_INVALID_ARG, "NULL kd, vd, dkd or dvd with L = %d", L);
  if (!(scale > 0.f) || scale == __builtin_inff())
    return fail(MODA_ERR_INVALID_ARG, "scale must be positive and finite");
  const int G = Hq / Hk;
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(MODA_ERR_UNSUPPORTED, "G = Hq/Hk = %d (supported: 1, 2, 4, 8, 16)", G);
  if (T > (1 << 24)) return fail(MODA_ERR_UNSUPPORTED, "T = %d > 2^24", T);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  const void* all[] = {q, k, v, o, lse, dO, dq, dk, dv, delta, L ? kd : nullptr, L ? vd : nullptr,
                       L ? dkd : nullptr, L ? dvd : nullptr};
  for (const void* p : all)
    if (p && !aligned16(p)) return fail(MODA_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  const size_t qb = (size_t)T * Hq * d * 2, kvb = (size_t)T * Hk * d * 2;
  const size_t db = (size_t)Hk * T * L * d * 2, lb = (size_t)T * Hq * 4;
  const void* ins[] = {q, k, v, L ? kd : nullptr, L ? vd : nullptr, o, lse, dO};
  const size_t insz[] = {qb, kvb, kvb, db, db, qb, lb, qb};
  void* outs[] = {dq, dk, dv, L ? dkd : nullptr, L ? dvd : nullptr, delta};
  const size_t outsz[] = {2 * qb, 2 * kvb, 2 * kvb, 2 * db, 2 * db, lb};
  for (int a = 0; a < 6; ++a) {
    for (int b = 0; b < 8; ++b)
      if (overlaps(outs[a], outsz[a], ins[b], insz[b]))
        return fail(MODA_ERR_INVALID_ARG, "an output or the workspace overlaps an input");
    for (int b = a + 1; b < 6; ++b)
      if (overlaps(outs[a], outsz[a], outs[b], outsz[b]))
        return fail(MODA_ERR_INVALID_ARG, "two outputs overlap");
  }
  moda::BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.kd = L ? kd : nullptr; a.vd = L ? vd : nullptr;
  a.o = o; a.dO = dO; a.lse = lse;
  a.T = T; a.Hq = Hq; a.Hk = Hk; a.d = d; a.L = L; a.G = G; a.scale = scale;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dkd = L ? dkd : nullptr; a.dvd = L ? dvd : nullptr;
  a.delta = delta;
  a.layer_major = layer_major;
  int dev;
  moda_status st = device_state(&dev, &a.err, &a.num_sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_bwd(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "moda_bwd launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_bwd(const void* q, const void* k, const void* v, const void* kd, const void* vd,
                     const void* o, const float* lse, const void* dO, int T, int Hq, int Hk,
                     int d, int L, float scale, float* dq, float* dk, float* dv, float* dkd,
                     float* dvd, float* delta, moda_stream_t stream) {
  return bwd_impl(q, k, v, kd, vd, o, lse, dO, T, Hq, Hk, d, L, scale, dq, dk, dv, dkd, dvd, delta,
                  stream, 0);
}

moda_status moda_bwd_layer_major(const void* q, const void* k, const void* v, const void* kd,
                                 const void* vd, const void* o, const float* lse, const void* dO,
                                 int T, int Hq, int Hk, int d, int L, float scale, float* dq,
                                 float* dk, float* dv, float* dkd, float* dvd, float* delta,
                                 moda_stream_t stream) {
  return bwd_impl(q, k, v, kd, vd, o, lse, dO, T, Hq, Hk, d, L, scale, dq, dk, dv, dkd, dvd, delta,
                  stream, 1);
}

size_t moda_decode_workspace_bytes(int Tctx, int Hq, int d) {
  if (Tctx < 1 || Hq < 1 || d < 1) return 0;
  return (size_t)(moda::decode_num_splits(Tctx) + 1) * Hq * (d + 2) * sizeof(float);
}

// slot_stride == 0: moda_decode's [L, d] blocks (consecutive slots d apart,
// blocks at least L*d apart); otherwise any slot and KV-head strides.
static moda_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                               const void* kd_tok, const void* vd_tok, long long slot_stride,
                               long long depth_hk_stride, int Tctx, int Hq, int Hk, int d, int L,
                               float scale, void* o, float* lse, float* workspace,
                               size_t workspace_bytes, moda_stream_t stream) {
  if (!q || !k_cache || !v_cache || !o || !workspace)
    return fail(MODA_ERR_INVALID_ARG, "NULL q, cache, o or workspace");
  if (Tctx < 1) return fail(MODA_ERR_INVALID_ARG, "Tctx = %d < 1", Tctx);
  if (L < 0) return fail(MODA_ERR_INVALID_ARG, "L = %d < 0", L);
  if (Hk < 1 || Hq < 1) return fail(MODA_ERR_INVALID_ARG, "Hq = %d, Hk = %d", Hq, Hk);
  if (Hq % Hk != 0) return fail(MODA_ERR_INVALID_ARG, "Hq = %d not a multiple of Hk = %d", Hq, Hk);
  if (L > 0 && (!kd_tok || !vd_tok)) return fail(MODA_ERR_INVALID_ARG, "NULL depth slots with L = %d", L);
  if (!(scale > 0.f) || scale == __builtin_inff())
    return fail(MODA_ERR_INVALID_ARG, "scale must be positive and finite");
  const int G = Hq / Hk;
  if (d != 64 && d != 128) return fail(MODA_ERR_UNSUPPORTED, "d = %d (supported: 64, 128)", d);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(MODA_ERR_UNSUPPORTED, "G = Hq/Hk = %d (supported: 1, 2, 4, 8, 16)", G);
  if (Tctx > (1 << 24)) return fail(MODA_ERR_UNSUPPORTED, "Tctx = %d > 2^24", Tctx);
  if (L > 1024) return fail(MODA_ERR_UNSUPPORTED, "L = %d > 1024", L);
  if (slot_stride == 0) {
    if (L > 0 && (depth_hk_stride < (long long)L * d || depth_hk_stride % 8 != 0))
      return fail(MODA_ERR_INVALID_ARG, "depth_hk_stride = %lld must be >= L*d and a multiple of 8",
                  depth_hk_stride);
    slot_stride = d;
  } else if (L > 0 && (slot_stride < d || slot_stride % 8 != 0 ||
                       (Hk > 1 && (depth_hk_stride < d || depth_hk_stride % 8 != 0)))) {
    return fail(MODA_ERR_INVALID_ARG,
                "depth strides (slot %lld, KV head %lld) must be >= d and multiples of 8",
                slot_stride, depth_hk_stride);
  }
  if (Hk == 1) depth_hk_stride = (long long)L * d;  // never used to step between heads
  if (workspace_bytes < moda_decode_workspace_bytes(Tctx, Hq, d))
    return fail(MODA_ERR_INVALID_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes,
                moda_decode_workspace_bytes(Tctx, Hq, d));
  const void* al[] = {q, k_cache, v_cache, o, workspace, lse, L ? kd_tok : nullptr, L ? vd_tok : nullptr};
  for (const void* p : al)
    if (p && !aligned16(p)) return fail(MODA_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  const size_t qb = (size_t)Hq * d * 2, cb = (size_t)Tctx * Hk * d * 2;
  const size_t db =
      L ? ((size_t)(Hk - 1) * depth_hk_stride + (size_t)(L - 1) * slot_stride + (size_t)d) * 2 : 0;
  const void* ins[] = {q, k_cache, v_cache, L ? kd_tok : nullptr, L ? vd_tok : nullptr};
  const size_t insz[] = {qb, cb, cb, db, db};
  void* outs[] = {o, lse, workspace};
  const size_t outsz[] = {qb, lse ? (size_t)Hq * 4 : 0, workspace_bytes};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 5; ++b)
      if (overlaps(outs[a], outsz[a], ins[b], insz[b]))
        return fail(MODA_ERR_INVALID_ARG, "an output or the workspace overlaps an input");
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(outs[a], outsz[a], outs[b], outsz[b]))
        return fail(MODA_ERR_INVALID_ARG, "outputs overlap");
  }
  moda::DecodeArgs a{};
  a.q = q; a.k = k_cache; a.v = v_cache; a.kd = L ? kd_tok : nullptr; a.vd = L ? vd_tok : nullptr;
  a.depth_hk_stride = depth_hk_stride;
  a.depth_slot_stride = slot_stride;
  a.Tctx = Tctx; a.Hq = Hq; a.Hk = Hk; a.d = d; a.L = L; a.G = G; a.scale = scale;
  a.o = o; a.lse = lse; a.work = workspace;
  int dev;
  moda_status st = device_state(&dev, &a.err, &a.num_sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_decode(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "moda_decode launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_decode(const void* q, const void* k_cache, const void* v_cache,
                        const void* kd_tok, const void* vd_tok, long long depth_hk_stride,
                        int Tctx, int Hq, int Hk, int d, int L, float scale, void* o, float* lse,
                        float* workspace, size_t workspace_bytes, moda_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, kd_tok, vd_tok, 0, depth_hk_stride, Tctx, Hq, Hk, d, L,
                     scale, o, lse, workspace, workspace_bytes, stream);
}

moda_status moda_decode_strided(const void* q, const void* k_cache, const void* v_cache,
                                const void* kd_tok, const void* vd_tok,
                                long long depth_slot_stride, long long depth_hk_stride, int Tctx,
                                int Hq, int Hk, int d, int L, float scale, void* o, float* lse,
                                float* workspace, size_t workspace_bytes, moda_stream_t stream) {
  if (L > 0 && depth_slot_stride < 1)
    return fail(MODA_ERR_INVALID_ARG, "depth_slot_stride = %lld < 1", depth_slot_stride);
  return decode_impl(q, k_cache, v_cache, kd_tok, vd_tok, L > 0 ? depth_slot_stride : d,
                     depth_hk_stride, Tctx, Hq, Hk, d, L, scale, o, lse, workspace,
                     workspace_bytes, stream);
}

moda_status moda_selftest_wait_timeout(int timeout_ms, moda_stream_t stream) {
  if (timeout_ms < 1 || timeout_ms > 5000)
    return fail(MODA_ERR_INVALID_ARG, "timeout_ms = %d (allowed 1..5000)", timeout_ms);
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  cudaError_t e = moda::launch_selftest_wait(err, timeout_ms, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
  return ok();
}

moda_status moda_get_device_error(moda_stream_t stream) {
  int dev, sms;
  unsigned int* err;
  moda_status st = device_state(&dev, &err, &sms);
  if (st != MODA_OK) return st;
  unsigned int val = 0;
  const unsigned int zero = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&val, err, sizeof val, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(err, &zero, sizeof zero, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MODA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  if (val != 0) return fail((moda_status)val, "a kernel latched %s", moda_status_string((moda_status)val));
  return ok();
}

}  // extern "C"
