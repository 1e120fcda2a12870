// C-ABI layer of libkda: argument validation, dispatch to the kernels, status
// codes and the per-device error word.  Declarations and the contract of every
// entry point are in include/kda.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "kda.h"
#include "kda_internal.h"
#include "kda_backward_chunk.h"

namespace {

thread_local std::string g_msg;

// Launch accounting of the calling thread (kda_set_launch_events,
// kda_last_launch_count).  `ev` is armed for one compute call.
struct LaunchLog {
  void* const* ev = nullptr;
  int cap = 0;
  int used = 0;
  int launches = 0;
  cudaError_t pending = cudaSuccess;  // a failed record of events[0]
};
thread_local LaunchLog g_launch;

// Scope of one compute call: resets the count, and disarms the events at exit.
struct LaunchScope {
  LaunchScope() {
    g_launch.launches = 0;
    g_launch.used = 0;
    g_launch.pending = cudaSuccess;
  }
  ~LaunchScope() {
    g_launch.ev = nullptr;
    g_launch.cap = 0;
  }
};

kda_status fail(kda_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return st;
}

// Device error word, one per device (a module-scope device variable is
// instantiated on every device that loads the library).
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

kda_status device_error_ptr(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(KDA_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess)
      return fail(KDA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return KDA_OK;
}

size_t esize(int32_t dt) {
  switch (dt) {
    case KDA_DTYPE_F32:
      return 4;
    case KDA_DTYPE_BF16:
      return 2;
    case KDA_DTYPE_I32:
      return 4;
    default:
      return 0;
  }
}

const char* dtname(int32_t dt) {
  switch (dt) {
    case KDA_DTYPE_F32:
      return "f32";
    case KDA_DTYPE_BF16:
      return "bf16";
    case KDA_DTYPE_I32:
      return "i32";
    default:
      return "?";
  }
}

struct Extent {
  uintptr_t lo = 0, hi = 0;  // [lo, hi); empty when lo == hi
};

Extent extent(const kda_tensor* t) {
  Extent e;
  if (!t || !t->data) return e;
  int64_t last = 0;
  for (int d = 0; d < t->ndim; ++d) {
    if (t->shape[d] == 0) return e;
    last += (t->shape[d] - 1) * t->stride[d];
  }
  const size_t es = esize(t->dtype);
  e.lo = reinterpret_cast<uintptr_t>(t->data);
  e.hi = e.lo + (uintptr_t)(last + 1) * es;
  return e;
}

bool overlap(const kda_tensor* a, const kda_tensor* b) {
  const Extent x = extent(a), y = extent(b);
  if (x.lo == x.hi || y.lo == y.hi) return false;
  return x.lo < y.hi && y.lo < x.hi;
}

// Checks a descriptor: rank, non-negative sizes and strides, innermost
// contiguity and alignment (`align` bytes for the pointer and outer strides).
kda_status check_desc(const kda_tensor* t, const char* name, int ndim, size_t align) {
  if (!t) return fail(KDA_ERR_INVALID_ARG, "%s: descriptor is NULL", name);
  if (t->ndim != ndim)
    return fail(KDA_ERR_INVALID_ARG, "%s: expected %d dimensions, got %d", name, ndim, t->ndim);
  const size_t es = esize(t->dtype);
  if (!es) return fail(KDA_ERR_INVALID_ARG, "%s: unknown dtype %d", name, t->dtype);
  int64_t numel = 1;
  for (int d = 0; d < ndim; ++d) {
    if (t->shape[d] < 0 || t->stride[d] < 0)
      return fail(KDA_ERR_INVALID_ARG, "%s: negative size or stride in dim %d", name, d);
    numel *= t->shape[d];
  }
  if (numel == 0) return KDA_OK;
  if (!t->data) return fail(KDA_ERR_INVALID_ARG, "%s: data is NULL", name);
  if (t->stride[ndim - 1] != 1 && t->shape[ndim - 1] > 1)
    return fail(KDA_ERR_INVALID_ARG, "%s: innermost stride must be 1", name);
  if (reinterpret_cast<uintptr_t>(t->data) % align)
    return fail(KDA_ERR_INVALID_ARG, "%s: data pointer not %zu-byte aligned", name, align);
  for (int d = 0; d + 1 < ndim; ++d)
    if (t->shape[d] > 1 && ((size_t)t->stride[d] * es) % align)
      return fail(KDA_ERR_INVALID_ARG, "%s: stride of dim %d is not a multiple of %zu bytes",
                  name, d, align);
  return KDA_OK;
}

kda_status check_shape(const kda_tensor* t, const char* name, int ndim, const int64_t* want,
                       int32_t dtype) {
  if (t->dtype != dtype)
    return fail(KDA_ERR_INVALID_ARG, "%s: dtype %s, expected %s", name, dtname(t->dtype),
                dtname(dtype));
  for (int d = 0; d < ndim; ++d)
    if (t->shape[d] != want[d])
      return fail(KDA_ERR_INVALID_ARG, "%s: size %lld in dim %d, expected %lld", name,
                  (long long)t->shape[d], d, (long long)want[d]);
  return KDA_OK;
}

#define KDA_TRY(x)                \
  do {                            \
    kda_status st_ = (x);         \
    if (st_ != KDA_OK) return st_; \
  } while (0)

kda_status check_head_dims(int64_t dk, int64_t dv) {
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128))
    return fail(KDA_ERR_UNSUPPORTED, "head dims d_k=%lld d_v=%lld; supported: 64, 128",
                (long long)dk, (long long)dv);
  return KDA_OK;
}

kda_status check_state(const kda_tensor* s, const char* name, int64_t N, int64_t H, int64_t dk,
                       int64_t dv) {
  KDA_TRY(check_desc(s, name, 4, 16));
  const int64_t want[4] = {N, H, dk, dv};
  KDA_TRY(check_shape(s, name, 4, want, KDA_DTYPE_F32));
  if (N * H > 0 && s->stride[2] != dv)
    return fail(KDA_ERR_INVALID_ARG, "%s: inner [d_k, d_v] block must be contiguous", name);
  return KDA_OK;
}

kda::Act act(const kda_tensor* t) {
  kda::Act a;
  a.ptr = t->data;
  if (t->ndim == 4) {
    a.sb = t->stride[0];
    a.st = t->stride[1];
    a.sh = t->stride[2];
  } else {  // [N, H, D]
    a.sb = t->stride[0];
    a.st = 0;
    a.sh = t->stride[1];
  }
  return a;
}

cudaMemPool_t g_pool[kMaxDevices];

kda_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Armed by kda_test_stall_next_prefill; consumed by the calling thread's next
// prefill call, whatever path it takes.
thread_local int g_test_stall = 0;

// Domain checks of a prefill-shaped argument set (KDA_VALIDATE), enqueued before
// the compute kernels.
cudaError_t validate_prefill(const kda::PrefillArgs& a, cudaStream_t st) {
  kda::ValidateArgs va;
  memset(&va, 0, sizeof(va));
  va.q = a.q;
  va.k = a.k;
  va.v = a.v;
  va.g = a.g;
  va.beta = a.beta;
  va.beta_sb = a.beta_sb;
  va.beta_st = a.beta_st;
  va.beta_sh = a.beta_sh;
  va.gate_scale = a.gate ? a.gate_scale : nullptr;
  va.B = a.B;
  va.T = a.T;
  va.H = a.H;
  va.dk = a.dk;
  va.dv = a.dv;
  va.bf16 = a.bf16;
  va.gate = a.gate;
  va.err = a.err;
  return kda::launch_validate(va, st);
}

// The same for one decode token per request: rows are the N requests.
cudaError_t validate_decode(const kda::DecodeArgs& d, int* err, cudaStream_t st) {
  kda::PrefillArgs a;
  memset(&a, 0, sizeof(a));
  a.q = d.q;
  a.k = d.k;
  a.v = d.v;
  a.g = d.g;
  a.q.st = a.k.st = a.v.st = a.g.st = 0;
  a.beta = d.beta;
  a.beta_sb = d.beta_sn;
  a.beta_sh = d.beta_sh;
  a.B = d.N;
  a.T = 1;
  a.H = d.H;
  a.dk = d.dk;
  a.dv = d.dv;
  a.bf16 = d.bf16;
  a.err = err;
  return validate_prefill(a, st);
}

enum class PrefillPath { kChunked, kRecurrent, kChunkedNoAlloc };

kda_status prefill(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                   const kda_tensor* g, const kda_tensor* beta, const kda_tensor* s0,
                   float scale, const kda_tensor* cu, kda_tensor* out, kda_tensor* sT,
                   void* stream, PrefillPath path, const kda_tensor* gate_scale = nullptr,
                   kda_tensor* ckpt = nullptr, int64_t ck_tokens = 0) {
  g_msg.clear();
  const int stall = g_test_stall;
  g_test_stall = 0;
  KDA_TRY(check_desc(q, "q", 4, 16));
  const int32_t dt = q->dtype;
  if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32)
    return fail(KDA_ERR_INVALID_ARG, "q: dtype must be bf16 or f32");
  const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2], dk = q->shape[3];
  KDA_TRY(check_desc(v, "v", 4, 16));
  const int64_t dv = v->shape[3];
  KDA_TRY(check_head_dims(dk, dv));
  const int64_t wq[4] = {B, T, H, dk}, wv[4] = {B, T, H, dv}, wb[3] = {B, T, H};
  KDA_TRY(check_desc(k, "k", 4, 16));
  KDA_TRY(check_shape(k, "k", 4, wq, dt));
  KDA_TRY(check_shape(v, "v", 4, wv, dt));
  const bool gated = gate_scale != nullptr;
  KDA_TRY(check_desc(g, gated ? "gate" : "g", 4, 16));
  KDA_TRY(check_shape(g, gated ? "gate" : "g", 4, wq, gated ? dt : KDA_DTYPE_F32));
  if (gated) {
    KDA_TRY(check_desc(gate_scale, "gate_scale", 1, 4));
    const int64_t wh[1] = {H};
    KDA_TRY(check_shape(gate_scale, "gate_scale", 1, wh, KDA_DTYPE_F32));
  }
  KDA_TRY(check_desc(beta, "beta", 3, 4));
  KDA_TRY(check_shape(beta, "beta", 3, wb, KDA_DTYPE_F32));
  KDA_TRY(check_desc(out, "out", 4, 16));
  KDA_TRY(check_shape(out, "out", 4, wv, dt));
  if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (T > INT32_MAX || B > INT32_MAX || H > 65535)
    return fail(KDA_ERR_UNSUPPORTED, "sizes too large (T, B < 2^31, H < 65536)");
  int64_t N = B;
  if (cu) {
    KDA_TRY(check_desc(cu, "cu_seqlens", 1, 4));
    if (cu->dtype != KDA_DTYPE_I32) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: dtype must be i32");
    if (cu->shape[0] < 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: needs N+1 >= 1 entries");
    if (B != 1) return fail(KDA_ERR_INVALID_ARG, "varlen (cu_seqlens) requires B == 1, got %lld",
                            (long long)B);
    N = cu->shape[0] - 1;
  }
  if (N * H > INT32_MAX / 8) return fail(KDA_ERR_UNSUPPORTED, "too many (sequence, head) pairs");
  if (s0) KDA_TRY(check_state(s0, "initial_state", N, H, dk, dv));
  if (sT) KDA_TRY(check_state(sT, "final_state", N, H, dk, dv));
  // aliasing
  const kda_tensor* ins[] = {q, k, v, g, beta, s0, cu, gate_scale};
  const char* in_names[] = {"q", "k", "v", "g", "beta", "initial_state", "cu_seqlens", "gate_scale"};
  for (int i = 0; i < 8; ++i)
    if (ins[i] && overlap(out, ins[i]))
      return fail(KDA_ERR_INVALID_ARG, "out overlaps %s", in_names[i]);
  if (sT && gate_scale && overlap(sT, gate_scale))
    return fail(KDA_ERR_INVALID_ARG, "final_state overlaps gate_scale");
  int64_t ck_count = 0;
  if (ckpt) {
    if (ck_tokens <= 0 || ck_tokens % 64 != 0 || ck_tokens > INT32_MAX)
      return fail(KDA_ERR_INVALID_ARG, "checkpoint_tokens must be a positive multiple of 64, got %lld",
                  (long long)ck_tokens);
    KDA_TRY(check_desc(ckpt, "checkpoints", 4, 16));
    if (ckpt->dtype != KDA_DTYPE_F32) return fail(KDA_ERR_INVALID_ARG, "checkpoints: dtype must be f32");
    if (N > 0 && ckpt->shape[0] % N != 0)
      return fail(KDA_ERR_INVALID_ARG, "checkpoints: %lld rows is not a multiple of N = %lld",
                  (long long)ckpt->shape[0], (long long)N);
    ck_count = N > 0 ? ckpt->shape[0] / N : 0;
    if (ckpt->shape[1] != H || ckpt->shape[2] != dk || ckpt->shape[3] != dv)
      return fail(KDA_ERR_INVALID_ARG, "checkpoints: expected [N * C, %lld, %lld, %lld]", (long long)H,
                  (long long)dk, (long long)dv);
    if (ckpt->stride[2] != dv)
      return fail(KDA_ERR_INVALID_ARG, "checkpoints: inner [d_k, d_v] block must be contiguous");
    if (ck_count > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many checkpoints");
    const kda_tensor* others[] = {q, k, v, g, beta, s0, cu, gate_scale, out, sT};
    const char* onames[] = {"q", "k", "v", "g", "beta", "initial_state", "cu_seqlens", "gate_scale", "out",
                            "final_state"};
    for (int i = 0; i < 10; ++i)
      if (others[i] && overlap(ckpt, others[i]))
        return fail(KDA_ERR_INVALID_ARG, "checkpoints overlaps %s", onames[i]);
  }
  if (sT) {
    if (overlap(out, sT)) return fail(KDA_ERR_INVALID_ARG, "out overlaps final_state");
    for (int i = 0; i < 5; ++i)
      if (overlap(sT, ins[i])) return fail(KDA_ERR_INVALID_ARG, "final_state overlaps %s", in_names[i]);
    if (cu && overlap(sT, cu)) return fail(KDA_ERR_INVALID_ARG, "final_state overlaps cu_seqlens");
    if (s0 && overlap(sT, s0)) {
      const bool same = s0->data == sT->data && s0->stride[0] == sT->stride[0] &&
                        s0->stride[1] == sT->stride[1];
      if (!same)
        return fail(KDA_ERR_INVALID_ARG, "final_state partly overlaps initial_state");
    }
  }

  kda::PrefillArgs a;
  memset(&a, 0, sizeof(a));
  a.q = act(q);
  a.k = act(k);
  a.v = act(v);
  a.g = act(g);
  a.beta = static_cast<const float*>(beta->data);
  a.beta_sb = beta->stride[0];
  a.beta_st = beta->stride[1];
  a.beta_sh = beta->stride[2];
  if (s0 && N * H > 0) {
    a.s0 = static_cast<const float*>(s0->data);
    a.s0_sn = s0->stride[0];
    a.s0_sh = s0->stride[1];
  }
  if (sT && N * H > 0) {
    a.sT = static_cast<float*>(sT->data);
    a.sT_sn = sT->stride[0];
    a.sT_sh = sT->stride[1];
  }
  a.out = out->data;
  a.out_sb = out->stride[0];
  a.out_st = out->stride[1];
  a.out_sh = out->stride[2];
  a.cu_seqlens = cu ? static_cast<const int32_t*>(cu->data) : nullptr;
  a.B = (int)B;
  a.T = (int)T;
  a.H = (int)H;
  a.N = (int)N;
  a.dk = (int)dk;
  a.dv = (int)dv;
  a.bf16 = dt == KDA_DTYPE_BF16;
  a.scale = scale;
  a.gate = gated ? 1 : 0;
  a.gate_scale = gated ? static_cast<const float*>(gate_scale->data) : nullptr;
  if (ckpt && ck_count > 0 && H > 0) {
    a.ckpt = static_cast<float*>(ckpt->data);
    a.ck_sr = ckpt->stride[0];
    a.ck_sh = ckpt->stride[1];
    a.ck_count = (int)ck_count;
    a.ck_tokens = (int)ck_tokens;
  }
  if (N * H == 0) return KDA_OK;
  if (!a.sT && T == 0) return KDA_OK;
  if (path == PrefillPath::kChunkedNoAlloc && a.bf16) {
    const size_t need = kda::chunk_prefill_workspace_bytes(a);
    if (need > kda::kNoallocWorkspaceBytes)
      return fail(KDA_ERR_UNSUPPORTED,
                  "this call needs %zu bytes of chunk-record scratch but the fixed workspace of "
                  "kda_chunk_fwd_noalloc holds %zu; split the batch or use kda_chunk_fwd",
                  need, (size_t)kda::kNoallocWorkspaceBytes);
  }
  a.test_stall = stall;
  KDA_TRY(device_error_ptr(&a.err));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kda::validate_enabled() && (e = validate_prefill(a, st)) != cudaSuccess)
    return cuda_fail(e, "input check launch");
  void* fixed_ws = nullptr;
  if (path == PrefillPath::kChunkedNoAlloc && a.bf16) {
    e = kda::noalloc_workspace(&fixed_ws);
    if (e != cudaSuccess) return cuda_fail(e, "fixed workspace address lookup");
  }
  if (cu) {
    e = kda::launch_check_seqlens(a.cu_seqlens, a.N, a.T, a.err, st);
    if (e != cudaSuccess) return cuda_fail(e, "cu_seqlens check launch");
  }
  if (path == PrefillPath::kChunked && a.bf16) {
    const size_t ws_bytes = kda::chunk_prefill_workspace_bytes(a);
    void* ws = nullptr;
    if (ws_bytes) {
      e = kda::scratch_alloc(&ws, ws_bytes, st);
      if (e != cudaSuccess) return cuda_fail(e, "chunk-record workspace allocation");
    }
    e = kda::launch_chunk_prefill_tc(a, ws, st);
    const cudaError_t ef = ws ? kda::scratch_free(ws, st) : cudaSuccess;
    if (e == cudaSuccess) e = ef;
  } else if (path == PrefillPath::kChunkedNoAlloc && a.bf16) {
    e = kda::launch_chunk_prefill_tc(a, fixed_ws, st);
  } else {
    e = kda::launch_recurrent_prefill(a, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return KDA_OK;
}

}  // namespace

namespace kda {

void launch_begin(cudaStream_t s) {
  if (g_launch.ev && g_launch.used == 0 && g_launch.cap > 0) {
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(g_launch.ev[0]), s);
    if (e == cudaSuccess) {
      g_launch.used = 1;
    } else {  // reported by launch_end, not by the kernel's own launch check
      cudaGetLastError();
      g_launch.pending = e;
      g_launch.ev = nullptr;
    }
  }
}

cudaError_t launch_end(cudaStream_t s) {
  ++g_launch.launches;
  if (g_launch.pending != cudaSuccess) {
    const cudaError_t e = g_launch.pending;
    g_launch.pending = cudaSuccess;
    return e;
  }
  if (!g_launch.ev || g_launch.used == 0 || g_launch.used >= g_launch.cap) return cudaSuccess;
  cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(g_launch.ev[g_launch.used]), s);
  if (e != cudaSuccess) {
    cudaGetLastError();  // not sticky; the kernel's own launch check has already passed
    g_launch.ev = nullptr;
    return e;
  }
  ++g_launch.used;
  return cudaSuccess;
}

// Per-device pool that keeps freed blocks for reuse (release threshold: never),
// so repeated calls do not go back to the driver for their chunk records.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_pool[dev]) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t pool;
      e = cudaMemPoolCreate(&pool, &props);
      if (e != cudaSuccess) return e;
      uint64_t keep = ~0ull;
      e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      if (e != cudaSuccess) return e;
      g_pool[dev] = pool;
    }
  }
  return cudaMallocFromPoolAsync(p, bytes, g_pool[dev], s);
}

cudaError_t scratch_free(void* p, cudaStream_t s) { return cudaFreeAsync(p, s); }

}  // namespace kda

extern "C" {

kda_status kda_chunk_fwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta,
                         const kda_tensor* initial_state, float scale,
                         const kda_tensor* cu_seqlens, kda_tensor* out,
                         kda_tensor* final_state, void* stream) {
  LaunchScope scope;
  return prefill(q, k, v, g, beta, initial_state, scale, cu_seqlens, out, final_state, stream,
                 PrefillPath::kChunked);
}

kda_status kda_chunk_fwd_gated(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                               const kda_tensor* gate, const kda_tensor* gate_scale,
                               const kda_tensor* beta, const kda_tensor* initial_state, float scale,
                               const kda_tensor* cu_seqlens, kda_tensor* out,
                               kda_tensor* final_state, void* stream) {
  LaunchScope scope;
  if (!gate_scale) {
    g_msg.clear();
    return fail(KDA_ERR_INVALID_ARG, "gate_scale: descriptor is NULL");
  }
  return prefill(q, k, v, gate, beta, initial_state, scale, cu_seqlens, out, final_state, stream,
                 PrefillPath::kChunked, gate_scale);
}

kda_status kda_chunk_fwd_checkpointed(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                      const kda_tensor* g, const kda_tensor* beta,
                                      const kda_tensor* initial_state, float scale,
                                      const kda_tensor* cu_seqlens, int64_t checkpoint_tokens,
                                      kda_tensor* checkpoints, kda_tensor* out, kda_tensor* final_state,
                                      void* stream) {
  LaunchScope scope;
  if (!checkpoints) {
    g_msg.clear();
    return fail(KDA_ERR_INVALID_ARG, "checkpoints: descriptor is NULL");
  }
  return prefill(q, k, v, g, beta, initial_state, scale, cu_seqlens, out, final_state, stream,
                 PrefillPath::kChunked, nullptr, checkpoints, checkpoint_tokens);
}

kda_status kda_chunk_fwd_noalloc(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                 const kda_tensor* g, const kda_tensor* beta,
                                 const kda_tensor* initial_state, float scale,
                                 const kda_tensor* cu_seqlens, kda_tensor* out,
                                 kda_tensor* final_state, void* stream) {
  LaunchScope scope;
  return prefill(q, k, v, g, beta, initial_state, scale, cu_seqlens, out, final_state, stream,
                 PrefillPath::kChunkedNoAlloc);
}

kda_status kda_fused_recurrent_fwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                   const kda_tensor* g, const kda_tensor* beta,
                                   const kda_tensor* initial_state, float scale,
                                   const kda_tensor* cu_seqlens, kda_tensor* out,
                                   kda_tensor* final_state, void* stream) {
  LaunchScope scope;
  return prefill(q, k, v, g, beta, initial_state, scale, cu_seqlens, out, final_state, stream,
                 PrefillPath::kRecurrent);
}

kda_status kda_recurrent_step(kda_tensor* state, const kda_tensor* q, const kda_tensor* k,
                              const kda_tensor* v, const kda_tensor* g, const kda_tensor* beta,
                              float scale, kda_tensor* out, void* stream) {
  LaunchScope scope;
  g_msg.clear();
  KDA_TRY(check_desc(q, "q", 3, 16));
  const int32_t dt = q->dtype;
  if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32)
    return fail(KDA_ERR_INVALID_ARG, "q: dtype must be bf16 or f32");
  const int64_t N = q->shape[0], H = q->shape[1], dk = q->shape[2];
  KDA_TRY(check_desc(v, "v", 3, 16));
  const int64_t dv = v->shape[2];
  KDA_TRY(check_head_dims(dk, dv));
  const int64_t wq[3] = {N, H, dk}, wv[3] = {N, H, dv}, wb[2] = {N, H};
  KDA_TRY(check_desc(k, "k", 3, 16));
  KDA_TRY(check_shape(k, "k", 3, wq, dt));
  KDA_TRY(check_shape(v, "v", 3, wv, dt));
  KDA_TRY(check_desc(g, "g", 3, 16));
  KDA_TRY(check_shape(g, "g", 3, wq, KDA_DTYPE_F32));
  KDA_TRY(check_desc(beta, "beta", 2, 4));
  KDA_TRY(check_shape(beta, "beta", 2, wb, KDA_DTYPE_F32));
  KDA_TRY(check_desc(out, "out", 3, 16));
  KDA_TRY(check_shape(out, "out", 3, wv, dt));
  KDA_TRY(check_state(state, "state", N, H, dk, dv));
  if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (N * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many (request, head) pairs");
  const kda_tensor* ins[] = {q, k, v, g, beta, state};
  const char* names[] = {"q", "k", "v", "g", "beta", "state"};
  for (int i = 0; i < 6; ++i)
    if (overlap(out, ins[i])) return fail(KDA_ERR_INVALID_ARG, "out overlaps %s", names[i]);
  for (int i = 0; i < 5; ++i)
    if (overlap(state, ins[i])) return fail(KDA_ERR_INVALID_ARG, "state overlaps %s", names[i]);
  if (N * H == 0) return KDA_OK;

  kda::DecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.state = static_cast<float*>(state->data);
  a.s_sn = state->stride[0];
  a.s_sh = state->stride[1];
  a.q = act(q);
  a.k = act(k);
  a.v = act(v);
  a.g = act(g);
  a.beta = static_cast<const float*>(beta->data);
  a.beta_sn = beta->stride[0];
  a.beta_sh = beta->stride[1];
  a.out = out->data;
  a.out_sn = out->stride[0];
  a.out_sh = out->stride[1];
  a.N = (int)N;
  a.H = (int)H;
  a.dk = (int)dk;
  a.dv = (int)dv;
  a.bf16 = dt == KDA_DTYPE_BF16;
  a.scale = scale;
  cudaError_t e;
  if (kda::validate_enabled()) {
    int* err = nullptr;
    KDA_TRY(device_error_ptr(&err));
    if ((e = validate_decode(a, err, static_cast<cudaStream_t>(stream))) != cudaSuccess)
      return cuda_fail(e, "input check launch");
  }
  e = kda::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KDA_OK;
}

namespace {

// kda_backward (token loop, chunked = false) and kda_chunk_bwd (chunked form)
kda_status backward_impl(bool chunked, const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta, const kda_tensor* initial_state,
                         float scale, const kda_tensor* cu, const kda_tensor* d_out,
                         const kda_tensor* d_final_state, kda_tensor* dq, kda_tensor* dk, kda_tensor* dv,
                         kda_tensor* dg, kda_tensor* dbeta, kda_tensor* d_initial_state, void* stream) {
  LaunchScope scope;
  g_msg.clear();
  KDA_TRY(check_desc(q, "q", 4, 16));
  const int32_t dt = q->dtype;
  if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32)
    return fail(KDA_ERR_INVALID_ARG, "q: dtype must be bf16 or f32");
  const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2], dk_ = q->shape[3];
  KDA_TRY(check_desc(v, "v", 4, 16));
  const int64_t dv_ = v->shape[3];
  KDA_TRY(check_head_dims(dk_, dv_));
  const int64_t wq[4] = {B, T, H, dk_}, wv[4] = {B, T, H, dv_}, wb[3] = {B, T, H};
  KDA_TRY(check_desc(k, "k", 4, 16));
  KDA_TRY(check_shape(k, "k", 4, wq, dt));
  KDA_TRY(check_shape(v, "v", 4, wv, dt));
  KDA_TRY(check_desc(g, "g", 4, 16));
  KDA_TRY(check_shape(g, "g", 4, wq, KDA_DTYPE_F32));
  KDA_TRY(check_desc(beta, "beta", 3, 4));
  KDA_TRY(check_shape(beta, "beta", 3, wb, KDA_DTYPE_F32));
  KDA_TRY(check_desc(d_out, "d_out", 4, 16));
  KDA_TRY(check_shape(d_out, "d_out", 4, wv, dt));
  kda_tensor* gq[4] = {dq, dk, dv, dg};
  const char* gn[4] = {"dq", "dk", "dv", "dg"};
  for (int i = 0; i < 4; ++i) {
    KDA_TRY(check_desc(gq[i], gn[i], 4, 16));
    KDA_TRY(check_shape(gq[i], gn[i], 4, i == 2 ? wv : wq, KDA_DTYPE_F32));
  }
  KDA_TRY(check_desc(dbeta, "dbeta", 3, 4));
  KDA_TRY(check_shape(dbeta, "dbeta", 3, wb, KDA_DTYPE_F32));
  if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (T > INT32_MAX || B > INT32_MAX || H > 65535)
    return fail(KDA_ERR_UNSUPPORTED, "sizes too large (T, B < 2^31, H < 65536)");
  int64_t N = B;
  if (cu) {
    KDA_TRY(check_desc(cu, "cu_seqlens", 1, 4));
    if (cu->dtype != KDA_DTYPE_I32) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: dtype must be i32");
    if (cu->shape[0] < 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: needs N+1 >= 1 entries");
    if (B != 1) return fail(KDA_ERR_INVALID_ARG, "varlen (cu_seqlens) requires B == 1, got %lld", (long long)B);
    N = cu->shape[0] - 1;
  }
  if (N * H > INT32_MAX / 8) return fail(KDA_ERR_UNSUPPORTED, "too many (sequence, head) pairs");
  if (chunked) {  // chunk indices are int in the chunked kernels
    const int64_t nck = (T + 63) / 64;
    if ((cu ? nck + N : nck * N) > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many 64-token chunks");
  }
  if (initial_state) KDA_TRY(check_state(initial_state, "initial_state", N, H, dk_, dv_));
  if (d_final_state) KDA_TRY(check_state(d_final_state, "d_final_state", N, H, dk_, dv_));
  if (d_initial_state) KDA_TRY(check_state(d_initial_state, "d_initial_state", N, H, dk_, dv_));
  const kda_tensor* ins[] = {q, k, v, g, beta, initial_state, cu, d_out, d_final_state};
  const char* in_names[] = {"q", "k", "v", "g", "beta", "initial_state", "cu_seqlens", "d_out", "d_final_state"};
  kda_tensor* outs[] = {dq, dk, dv, dg, dbeta, d_initial_state};
  const char* out_names[] = {"dq", "dk", "dv", "dg", "dbeta", "d_initial_state"};
  for (int o = 0; o < 6; ++o) {
    if (!outs[o]) continue;
    for (int i = 0; i < 9; ++i)
      if (ins[i] && overlap(outs[o], ins[i]))
        return fail(KDA_ERR_INVALID_ARG, "%s overlaps %s", out_names[o], in_names[i]);
    for (int p = o + 1; p < 6; ++p)
      if (outs[p] && overlap(outs[o], outs[p]))
        return fail(KDA_ERR_INVALID_ARG, "%s overlaps %s", out_names[o], out_names[p]);
  }
  if (N * H == 0) return KDA_OK;

  kda::BackwardArgs ba;
  memset(&ba, 0, sizeof(ba));
  kda::PrefillArgs& a = ba.f;
  a.q = act(q);
  a.k = act(k);
  a.v = act(v);
  a.g = act(g);
  a.beta = static_cast<const float*>(beta->data);
  a.beta_sb = beta->stride[0];
  a.beta_st = beta->stride[1];
  a.beta_sh = beta->stride[2];
  if (initial_state) {
    a.s0 = static_cast<const float*>(initial_state->data);
    a.s0_sn = initial_state->stride[0];
    a.s0_sh = initial_state->stride[1];
  }
  a.cu_seqlens = cu ? static_cast<const int32_t*>(cu->data) : nullptr;
  a.B = (int)B;
  a.T = (int)T;
  a.H = (int)H;
  a.N = (int)N;
  a.dk = (int)dk_;
  a.dv = (int)dv_;
  a.bf16 = dt == KDA_DTYPE_BF16;
  a.scale = scale;
  ba.dout = act(d_out);
  if (d_final_state) {
    ba.dsT = static_cast<const float*>(d_final_state->data);
    ba.dsT_sn = d_final_state->stride[0];
    ba.dsT_sh = d_final_state->stride[1];
  }
  auto gact = [](kda_tensor* t) {
    kda::GradAct x;
    x.ptr = static_cast<float*>(t->data);
    x.sb = t->stride[0];
    x.st = t->stride[1];
    x.sh = t->stride[2];
    return x;
  };
  ba.dq = gact(dq);
  ba.dk = gact(dk);
  ba.dv = gact(dv);
  ba.dg = gact(dg);
  ba.dbeta = static_cast<float*>(dbeta->data);
  ba.db_sb = dbeta->stride[0];
  ba.db_st = dbeta->stride[1];
  ba.db_sh = dbeta->stride[2];
  if (d_initial_state) {
    ba.ds0 = static_cast<float*>(d_initial_state->data);
    ba.ds0_sn = d_initial_state->stride[0];
    ba.ds0_sh = d_initial_state->stride[1];
  }
  ba.nblk = (int)((T + kda::kBwdBlock - 1) / kda::kBwdBlock);
  KDA_TRY(device_error_ptr(&a.err));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kda::validate_enabled() && (e = validate_prefill(a, st)) != cudaSuccess)
    return cuda_fail(e, "input check launch");
  if (cu) {
    e = kda::launch_check_seqlens(a.cu_seqlens, a.N, a.T, a.err, st);
    if (e != cudaSuccess) return cuda_fail(e, "cu_seqlens check launch");
  }
  if (chunked) {
    const size_t cb = kda::chunk_backward_workspace_bytes(a);
    void* cws = nullptr;
    e = kda::scratch_alloc(&cws, cb, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward workspace allocation");
    e = kda::launch_chunk_backward(ba, cws, st);
    const cudaError_t ef = kda::scratch_free(cws, st);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return KDA_OK;
  }
  const int64_t rows = (int64_t)a.B * a.T;
  const size_t ws_bytes = kda::backward_workspace_bytes(a.N, a.H, a.T, rows, a.dk, a.dv);
  void* ws = nullptr;
  if (ws_bytes) {
    e = kda::scratch_alloc(&ws, ws_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward workspace allocation");
  }
  ba.ck = static_cast<float*>(ws);
  ba.scr = ba.ck + (int64_t)a.N * a.H * ba.nblk * a.dk * a.dv;
  ba.part = kda::backward_value_slices(a.N, a.H, a.dv) == 4
                ? ba.scr + (int64_t)a.N * a.H * kda::kBwdBlock * a.dk * a.dv
                : nullptr;
  e = kda::launch_backward(ba, st);
  const cudaError_t ef = ws ? kda::scratch_free(ws, st) : cudaSuccess;
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return KDA_OK;
}

}  // namespace

kda_status kda_backward(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                        const kda_tensor* g, const kda_tensor* beta, const kda_tensor* initial_state,
                        float scale, const kda_tensor* cu, const kda_tensor* d_out,
                        const kda_tensor* d_final_state, kda_tensor* dq, kda_tensor* dk, kda_tensor* dv,
                        kda_tensor* dg, kda_tensor* dbeta, kda_tensor* d_initial_state, void* stream) {
  return backward_impl(false, q, k, v, g, beta, initial_state, scale, cu, d_out, d_final_state, dq, dk, dv, dg,
                       dbeta, d_initial_state, stream);
}

kda_status kda_chunk_bwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta, const kda_tensor* initial_state,
                         float scale, const kda_tensor* cu, const kda_tensor* d_out,
                         const kda_tensor* d_final_state, kda_tensor* dq, kda_tensor* dk, kda_tensor* dv,
                         kda_tensor* dg, kda_tensor* dbeta, kda_tensor* d_initial_state, void* stream) {
  return backward_impl(true, q, k, v, g, beta, initial_state, scale, cu, d_out, d_final_state, dq, dk, dv, dg,
                       dbeta, d_initial_state, stream);
}

kda_status kda_decode_step_fused(kda_tensor* state, kda_tensor* conv_q, kda_tensor* conv_k,
                                 kda_tensor* conv_v, const kda_tensor* q, const kda_tensor* k,
                                 const kda_tensor* v, const kda_tensor* w_q, const kda_tensor* w_k,
                                 const kda_tensor* w_v, const kda_tensor* g, const kda_tensor* beta,
                                 const kda_tensor* out_gate, const kda_tensor* norm_weight, float scale,
                                 float eps, kda_tensor* out, void* stream) {
  LaunchScope scope;
  g_msg.clear();
  KDA_TRY(check_desc(q, "q", 3, 16));
  const int32_t dt = q->dtype;
  if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32)
    return fail(KDA_ERR_INVALID_ARG, "q: dtype must be bf16 or f32");
  const int64_t N = q->shape[0], H = q->shape[1], dk = q->shape[2];
  KDA_TRY(check_desc(v, "v", 3, 16));
  const int64_t dv = v->shape[2];
  KDA_TRY(check_head_dims(dk, dv));
  const int64_t wq3[3] = {N, H, dk}, wv3[3] = {N, H, dv}, wb[2] = {N, H};
  KDA_TRY(check_desc(k, "k", 3, 16));
  KDA_TRY(check_shape(k, "k", 3, wq3, dt));
  KDA_TRY(check_shape(v, "v", 3, wv3, dt));
  KDA_TRY(check_desc(g, "g", 3, 16));
  KDA_TRY(check_shape(g, "g", 3, wq3, KDA_DTYPE_F32));
  KDA_TRY(check_desc(beta, "beta", 2, 4));
  KDA_TRY(check_shape(beta, "beta", 2, wb, KDA_DTYPE_F32));
  KDA_TRY(check_desc(out_gate, "out_gate", 3, 16));
  KDA_TRY(check_shape(out_gate, "out_gate", 3, wv3, dt));
  KDA_TRY(check_desc(out, "out", 3, 16));
  KDA_TRY(check_shape(out, "out", 3, wv3, dt));
  KDA_TRY(check_state(state, "state", N, H, dk, dv));
  const int64_t cqk[4] = {N, 3, H, dk}, cvs[4] = {N, 3, H, dv};
  // the kernels move channel pairs: caches aligned to two elements
  const size_t pair = dt == KDA_DTYPE_BF16 ? 4 : 8;
  KDA_TRY(check_desc(conv_q, "conv_q", 4, pair));
  KDA_TRY(check_shape(conv_q, "conv_q", 4, cqk, dt));
  KDA_TRY(check_desc(conv_k, "conv_k", 4, pair));
  KDA_TRY(check_shape(conv_k, "conv_k", 4, cqk, dt));
  KDA_TRY(check_desc(conv_v, "conv_v", 4, pair));
  KDA_TRY(check_shape(conv_v, "conv_v", 4, cvs, dt));
  const kda_tensor* ws[3] = {w_q, w_k, w_v};
  const char* wn[3] = {"w_q", "w_k", "w_v"};
  for (int i = 0; i < 3; ++i) {
    const int64_t d = i < 2 ? dk : dv;
    const int64_t shp[3] = {H, d, 4};
    KDA_TRY(check_desc(ws[i], wn[i], 3, 16));
    KDA_TRY(check_shape(ws[i], wn[i], 3, shp, KDA_DTYPE_F32));
    if (ws[i]->stride[1] != 4 || ws[i]->stride[0] != 4 * d)
      return fail(KDA_ERR_INVALID_ARG, "%s: must be contiguous [H, d, 4]", wn[i]);
  }
  if (norm_weight) {
    const int64_t shp[1] = {dv};
    KDA_TRY(check_desc(norm_weight, "norm_weight", 1, 16));
    KDA_TRY(check_shape(norm_weight, "norm_weight", 1, shp, KDA_DTYPE_F32));
  }
  if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (!isfinite(eps) || eps < 0.f) return fail(KDA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (N * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many (request, head) pairs");
  const kda_tensor* ins[] = {q, k, v, g, beta, out_gate, w_q, w_k, w_v, norm_weight};
  const char* names[] = {"q", "k", "v", "g", "beta", "out_gate", "w_q", "w_k", "w_v", "norm_weight"};
  kda_tensor* outs[] = {state, conv_q, conv_k, conv_v, out};
  const char* onames[] = {"state", "conv_q", "conv_k", "conv_v", "out"};
  for (int o = 0; o < 5; ++o) {
    for (int i = 0; i < 10; ++i)
      if (ins[i] && overlap(outs[o], ins[i])) return fail(KDA_ERR_INVALID_ARG, "%s overlaps %s", onames[o], names[i]);
    for (int p = o + 1; p < 5; ++p)
      if (overlap(outs[o], outs[p])) return fail(KDA_ERR_INVALID_ARG, "%s overlaps %s", onames[o], onames[p]);
  }
  if (N * H == 0) return KDA_OK;

  kda::FusedDecodeArgs fa;
  memset(&fa, 0, sizeof(fa));
  kda::DecodeArgs& a = fa.d;
  a.state = static_cast<float*>(state->data);
  a.s_sn = state->stride[0];
  a.s_sh = state->stride[1];
  a.q = act(q);
  a.k = act(k);
  a.v = act(v);
  a.g = act(g);
  a.beta = static_cast<const float*>(beta->data);
  a.beta_sn = beta->stride[0];
  a.beta_sh = beta->stride[1];
  a.out = out->data;
  a.out_sn = out->stride[0];
  a.out_sh = out->stride[1];
  a.N = (int)N;
  a.H = (int)H;
  a.dk = (int)dk;
  a.dv = (int)dv;
  a.bf16 = dt == KDA_DTYPE_BF16;
  a.scale = scale;
  fa.cq = conv_q->data;
  fa.ck = conv_k->data;
  fa.cv = conv_v->data;
  fa.cq_sn = conv_q->stride[0]; fa.cq_ss = conv_q->stride[1]; fa.cq_sh = conv_q->stride[2];
  fa.ck_sn = conv_k->stride[0]; fa.ck_ss = conv_k->stride[1]; fa.ck_sh = conv_k->stride[2];
  fa.cv_sn = conv_v->stride[0]; fa.cv_ss = conv_v->stride[1]; fa.cv_sh = conv_v->stride[2];
  fa.wq = static_cast<const float*>(w_q->data);
  fa.wk = static_cast<const float*>(w_k->data);
  fa.wv = static_cast<const float*>(w_v->data);
  fa.gate = act(out_gate);
  fa.norm_w = norm_weight ? static_cast<const float*>(norm_weight->data) : nullptr;
  fa.eps = eps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kda::validate_enabled()) {  // g and beta as for the plain step; the raw q, k, v finite
    int* err = nullptr;
    KDA_TRY(device_error_ptr(&err));
    if ((e = validate_decode(a, err, st)) != cudaSuccess) return cuda_fail(e, "input check launch");
  }
  void* scratch = nullptr;
  e = kda::scratch_alloc(&scratch, kda::decode_fused_workspace_bytes(a.N, a.H, a.dk, a.dv), st);
  if (e != cudaSuccess) return cuda_fail(e, "fused decode workspace allocation");
  e = kda::launch_decode_fused(fa, scratch, st);
  const cudaError_t ef = kda::scratch_free(scratch, st);
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) return cuda_fail(e, "fused decode launch");
  return KDA_OK;
}

kda_status kda_recurrent_multi_step(kda_tensor* state, const kda_tensor* q, const kda_tensor* k,
                                    const kda_tensor* v, const kda_tensor* g, const kda_tensor* beta,
                                    float scale, const kda_tensor* num_accepted, kda_tensor* out,
                                    void* stream) {
  LaunchScope scope;
  g_msg.clear();
  KDA_TRY(check_desc(k, "k", 4, 16));
  const int32_t dt = k->dtype;
  if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32)
    return fail(KDA_ERR_INVALID_ARG, "k: dtype must be bf16 or f32");
  const int64_t N = k->shape[0], n = k->shape[1], H = k->shape[2], dk = k->shape[3];
  KDA_TRY(check_desc(v, "v", 4, 16));
  const int64_t dv = v->shape[3];
  KDA_TRY(check_head_dims(dk, dv));
  const int64_t wq[4] = {N, n, H, dk}, wv[4] = {N, n, H, dv}, wb[3] = {N, n, H};
  KDA_TRY(check_shape(v, "v", 4, wv, dt));
  KDA_TRY(check_desc(g, "g", 4, 16));
  KDA_TRY(check_shape(g, "g", 4, wq, KDA_DTYPE_F32));
  KDA_TRY(check_desc(beta, "beta", 3, 4));
  KDA_TRY(check_shape(beta, "beta", 3, wb, KDA_DTYPE_F32));
  if ((q == nullptr) != (out == nullptr))
    return fail(KDA_ERR_INVALID_ARG, "q and out must both be given or both be NULL");
  if (q) {
    KDA_TRY(check_desc(q, "q", 4, 16));
    KDA_TRY(check_shape(q, "q", 4, wq, dt));
    KDA_TRY(check_desc(out, "out", 4, 16));
    KDA_TRY(check_shape(out, "out", 4, wv, dt));
  }
  KDA_TRY(check_state(state, "state", N, H, dk, dv));
  if (num_accepted) {
    KDA_TRY(check_desc(num_accepted, "num_accepted", 1, 4));
    if (num_accepted->dtype != KDA_DTYPE_I32)
      return fail(KDA_ERR_INVALID_ARG, "num_accepted: dtype must be i32");
    if (num_accepted->shape[0] != N)
      return fail(KDA_ERR_INVALID_ARG, "num_accepted: %lld entries, expected %lld",
                  (long long)num_accepted->shape[0], (long long)N);
  }
  if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (n > INT32_MAX || N > INT32_MAX || H > 65535 || N * H > INT32_MAX / 8)
    return fail(KDA_ERR_UNSUPPORTED, "sizes too large");
  const kda_tensor* ins[] = {q, k, v, g, beta, num_accepted};
  const char* names[] = {"q", "k", "v", "g", "beta", "num_accepted"};
  for (int i = 0; i < 6; ++i) {
    if (!ins[i]) continue;
    if (overlap(state, ins[i])) return fail(KDA_ERR_INVALID_ARG, "state overlaps %s", names[i]);
    if (out && overlap(out, ins[i])) return fail(KDA_ERR_INVALID_ARG, "out overlaps %s", names[i]);
  }
  if (out && overlap(out, state)) return fail(KDA_ERR_INVALID_ARG, "out overlaps state");
  if (N * H == 0 || n == 0) return KDA_OK;

  kda::PrefillArgs a;
  memset(&a, 0, sizeof(a));
  if (q) a.q = act(q);
  a.k = act(k);
  a.v = act(v);
  a.g = act(g);
  a.beta = static_cast<const float*>(beta->data);
  a.beta_sb = beta->stride[0];
  a.beta_st = beta->stride[1];
  a.beta_sh = beta->stride[2];
  a.s0 = static_cast<const float*>(state->data);
  a.s0_sn = state->stride[0];
  a.s0_sh = state->stride[1];
  a.sT = static_cast<float*>(state->data);
  a.sT_sn = state->stride[0];
  a.sT_sh = state->stride[1];
  if (out) {
    a.out = out->data;
    a.out_sb = out->stride[0];
    a.out_st = out->stride[1];
    a.out_sh = out->stride[2];
  }
  a.accepted = num_accepted ? static_cast<const int32_t*>(num_accepted->data) : nullptr;
  a.B = (int)N;
  a.T = (int)n;
  a.H = (int)H;
  a.N = (int)N;
  a.dk = (int)dk;
  a.dv = (int)dv;
  a.bf16 = dt == KDA_DTYPE_BF16;
  a.scale = scale;
  KDA_TRY(device_error_ptr(&a.err));
  cudaError_t e;
  if (kda::validate_enabled() && (e = validate_prefill(a, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "input check launch");
  e = kda::launch_recurrent_prefill(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "multi-step decode launch");
  return KDA_OK;
}

kda_status kda_get_device_error(void* stream) {
  g_msg.clear();
  int* p = nullptr;
  KDA_TRY(device_error_ptr(&p));
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word == 0) return KDA_OK;
  const int zero = 0;
  e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  if (word & kda::kErrTimeout)
    return fail(KDA_ERR_TIMEOUT, "a bounded device-side wait gave up (word 0x%x)", word);
  if (word & kda::kErrBadSeqlens)
    return fail(KDA_ERR_DEVICE, "cu_seqlens must start at 0, never decrease and end at T (word 0x%x)",
                word);
  return fail(KDA_ERR_DOMAIN,
              "an input is outside its domain: q, k, v finite, g in [-5, 0], beta in [0, 1] (word 0x%x)",
              word);
}

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK:
      return "KDA_OK";
    case KDA_ERR_INVALID_ARG:
      return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED:
      return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA:
      return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE:
      return "KDA_ERR_DEVICE";
    case KDA_ERR_TIMEOUT:
      return "KDA_ERR_TIMEOUT";
    case KDA_ERR_DOMAIN:
      return "KDA_ERR_DOMAIN";
  }
  return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error_message(void) { return g_msg.c_str(); }

kda_status kda_set_launch_events(void* const* events, int count) {
  g_msg.clear();
  if (count < 0 || (!events && count > 0))
    return fail(KDA_ERR_INVALID_ARG, "launch events: %d handles at %p", count, (const void*)events);
  g_launch.ev = count > 0 ? events : nullptr;
  g_launch.cap = count;
  return KDA_OK;
}

int kda_last_launch_count(void) { return g_launch.launches; }

kda_status kda_test_stall_next_prefill(int on) {
  g_msg.clear();
  g_test_stall = on ? 1 : 0;
  return KDA_OK;
}

}  // extern "C"
