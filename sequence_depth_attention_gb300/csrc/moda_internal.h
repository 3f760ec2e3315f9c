// Internal declarations shared by the translation units of libmoda.so.
// Not part of the public ABI (that is include/moda.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moda.h"

namespace moda {

// Arguments of one forward call after validation on the host.
struct FwdArgs {
  const void* q;   // [T, Hq, d]
  const void* k;   // [T, Hk, d]
  const void* v;   // [T, Hk, d]
  const void* kd;  // [Hk, T, L, d] packed (or [L, T, Hk, d] when layer_major), nullptr when L == 0
  const void* vd;  // same layout as kd
  int T, Hq, Hk, d, L, G;
  int layer_major;  // kd/vd as the layers wrote them: [L, T, Hk, d]
  float scale;
  void* o;         // [T, Hq, d] bf16
  float* lse;      // [T, Hq] fp32 or nullptr
  unsigned int* err;  // device error word of the current device
  unsigned int* queue;  // {next tile, CTAs finished}, zero at launch, zero again at exit
  int num_sms;
  int device;
};

// Arguments of one backward call after validation on the host.
struct BwdArgs {
  const void *q, *k, *v, *kd, *vd, *o, *dO;  // bf16; kd/vd packed, nullptr when L == 0
  const float* lse;                          // [T, Hq]
  int T, Hq, Hk, d, L, G;
  float scale;
  float *dq, *dk, *dv, *dkd, *dvd;           // fp32 outputs (dkd/dvd packed)
  float* delta;                              // [T, Hq] caller workspace
  unsigned int* err;                         // device error word of the current device
  int num_sms;
  int layer_major;  // kd/vd and dkd/dvd as [L, T, Hk, d] instead of packed
};

// Arguments of one decode call after validation on the host.
struct DecodeArgs {
  const void *q, *k, *v, *kd, *vd;  // q [Hq,d]; k/v cache [Tctx,Hk,d]; depth slots (see stride)
  int64_t depth_hk_stride;           // elements between the [L,d] blocks of consecutive KV heads
  int64_t depth_slot_stride;         // elements between consecutive slots of one KV head
  int Tctx, Hq, Hk, d, L, G;
  float scale;
  void* o;                           // [Hq,d] bf16
  float* lse;                        // [Hq] or nullptr
  float* work;                       // partials, decode_workspace_floats
  unsigned int* err;                 // device error word
  int num_sms;
};
int decode_num_splits(int Tctx);

// Arguments of one depth-KV projection after validation on the host.
struct KvProjArgs {
  const void *x, *wk, *wv;  // x [T, Dm]; wk, wv [Hk*d, Dm] (bf16)
  int T, Dm, Hk, d, L, slot;
  void *kd, *vd;            // packed [Hk, T, L, d] bf16; slot `slot` is written
  unsigned int* err;
  int num_sms;
};

// Kernel error codes latched into the device error word (first one wins).
enum : unsigned int { kErrNone = 0, kErrTimeout = MODA_ERR_TIMEOUT };

// The calling thread's current CUDA context (nullptr if none is bound):
// device addresses of module variables are valid only in the context they
// were looked up in.
void* current_context();

// The current device after checking that it is an sm_103 part; otherwise
// MODA_ERR_NO_DEVICE (or MODA_ERR_CUDA) with the detail set.
moda_status checked_device(int* dev);

// Sets the calling thread's last-error detail (see moda_last_error_detail)
// and returns s.
moda_status report(moda_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));

// Launchers. Return cudaSuccess or the launch error.
cudaError_t launch_pack_depth(const void* src, void* dst, int L, int T, int Hk,
                              int d, cudaStream_t stream);
cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t stream);
// d = 64: two query tiles per CTA in ping-pong.
cudaError_t launch_fwd_pp(const FwdArgs& a, cudaStream_t stream);
// Depth part on CUDA cores, merged into o and lse that hold the L = 0 result.
cudaError_t launch_fwd_depth_cc(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
// The sequence share of dq on tcgen05, added to what the depth kernel wrote
// (L > 0) or written (L == 0).
cudaError_t launch_bwd_dq_tc(const BwdArgs& a, cudaStream_t stream);
// dk and dv of the sequence keys on tcgen05.
cudaError_t launch_bwd_dkdv_tc(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_kv_proj(const KvProjArgs& a, cudaStream_t stream);
// slot_dev non-null: the slot index is read from device memory (see
// depth_write.cu); err is the device error word.
cudaError_t launch_depth_write(const void* src, void* dst, int T, int Hk, int d, int L, int slot,
                               const int* slot_dev, unsigned int* err, int num_sms,
                               cudaStream_t stream);

// Arguments of one depth-mass call after validation on the host.
struct DepthMassArgs {
  const void *q, *kd;  // q [T,Hq,d]; kd packed [Hk,T,L,d] (bf16)
  const float* lse;    // [T,Hq], natural log, from moda_fwd
  int T, Hq, Hk, d, L, G;
  float scale;
  float* mass;         // [Hk, L] output
  float* work;         // depth_mass_workspace_floats(T, Hk, L) floats
};
size_t depth_mass_workspace_floats(int T, int Hk, int L);
cudaError_t launch_depth_mass(const DepthMassArgs& a, cudaStream_t stream);
cudaError_t launch_cache_admit(int* ages, const float* mass, int Hk, int S, int recent,
                               int new_age, int* slot_out, cudaStream_t stream);
cudaError_t launch_selftest_wait(unsigned int* err, int timeout_ms, cudaStream_t stream);

}  // namespace moda
