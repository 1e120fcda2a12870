// Input-domain checks, run before the compute kernels when KDA_VALIDATE is set in
// the environment.
//
// The chunked kernels form every decay exponent as a difference of cumulative
// log-decays inside a 16-token sub-block, which stays representable only while the
// per-token log-decay g lies in [-5, 0] (the lower-bounded decay of "Kimi K3
// 技术报告解读" (marsggbo.github.io) §3.5; beta is a sigmoid, so in [0, 1]).  A
// caller outside that domain gets a result that follows the recurrence's
// definition but may lose precision.  This kernel lets a caller find such inputs:
// it reads q, k, v, g (or the gate logits) and beta once and sets kErrDomain in the
// device error word if any value is not finite, any g is outside [-5, 0] or any
// beta outside [0, 1].  It never traps and changes nothing else.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kValidateThreads = 256;

template <bool BF16>
__device__ __forceinline__ float act_at(const Act& x, int64_t b, int64_t t, int64_t h, int c) {
  const int64_t off = b * x.sb + t * x.st + h * x.sh + c;
  if constexpr (BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(x.ptr)[off]);
  return static_cast<const float*>(x.ptr)[off];
}

// One warp per (batch row, token, head); lanes stride over the channels.
template <bool BF16>
__global__ void __launch_bounds__(kValidateThreads) kda_validate_kernel(ValidateArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.B * a.T * a.H;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool bad = false;
  for (int64_t r = w0; r < rows; r += nw) {
    const int64_t h = r % a.H, bt = r / a.H;
    const int64_t t = bt % a.T, b = bt / a.T;
    for (int c = lane; c < a.dk; c += 32) {
      const float qv = a.q.ptr ? act_at<BF16>(a.q, b, t, h, c) : 0.f;  // no q: state-only multi-step
      const float kv = act_at<BF16>(a.k, b, t, h, c);
      bad |= !isfinite(qv) || !isfinite(kv);
      if (a.gate) {
        bad |= !isfinite(act_at<BF16>(a.g, b, t, h, c));  // decay logits: any finite value
      } else {
        const float gv = act_at<false>(a.g, b, t, h, c);
        bad |= !(gv >= -5.f && gv <= 0.f);  // false for NaN as well
      }
    }
    for (int c = lane; c < a.dv; c += 32) bad |= !isfinite(act_at<BF16>(a.v, b, t, h, c));
    if (lane == 0) {
      const float be = a.beta[b * a.beta_sb + t * a.beta_st + h * a.beta_sh];
      bad |= !(be >= 0.f && be <= 1.f);
    }
  }
  if (a.gate_scale && blockIdx.x == 0 && threadIdx.x < 32)
    for (int h = lane; h < a.H; h += 32) bad |= !isfinite(a.gate_scale[h]);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, kErrDomain);
}

}  // namespace

bool validate_enabled() {
  const char* v = getenv("KDA_VALIDATE");
  return v && v[0] && !(v[0] == '0' && v[1] == 0);
}

cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s) {
  const int64_t rows = (int64_t)a.B * a.T * a.H;
  if (rows == 0 && !a.gate_scale) return cudaSuccess;
  const int64_t want = (rows * 32 + kValidateThreads - 1) / kValidateThreads;
  const int64_t cap = (int64_t)sm_count() * 8;
  const int grid = (int)(want < 1 ? 1 : (want < cap ? want : cap));
  launch_begin(s);
  if (a.bf16)
    kda_validate_kernel<true><<<grid, kValidateThreads, 0, s>>>(a);
  else
    kda_validate_kernel<false><<<grid, kValidateThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_end(s);
}

}  // namespace kda
