// Chunked backward of the KDA core: kernels and launcher.  The kernel bodies and
// the derivation they follow are in kda_backward_chunk.cuh.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_backward_chunk.cuh"
#include "kda_backward_chunk.h"

namespace kda {
namespace {

using bwdc::ChunkBwdArgs;
using bwdc::kC;
using bwdc::kW;

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(256, 1) kda_bwd_prep_kernel(ChunkBwdArgs ca) {
  extern __shared__ __align__(16) float sm[];
  bwdc::prep_body<DK, DV, T>(ca, sm, blockIdx.x, blockIdx.y, threadIdx.x);
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(bwdc::kPassThreads, 1) kda_bwd_state_fwd_kernel(ChunkBwdArgs ca) {
  extern __shared__ __align__(16) float sm[];
  bwdc::pass_body<DK, DV, T, false>(ca, sm, blockIdx.x, threadIdx.x);
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(bwdc::kPassThreads, 1) kda_bwd_state_rev_kernel(ChunkBwdArgs ca) {
  extern __shared__ __align__(16) float sm[];
  bwdc::pass_body<DK, DV, T, true>(ca, sm, blockIdx.x, threadIdx.x);
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(256, 1) kda_bwd_grad_kernel(ChunkBwdArgs ca) {
  extern __shared__ __align__(16) float sm[];
  bwdc::grad_body<DK, DV, T>(ca, sm, blockIdx.x, blockIdx.y, threadIdx.x);
}

// off[n] = number of chunks of the sequences before n (varlen), capped at `total`
__global__ void __launch_bounds__(1024) kda_bwd_offsets_kernel(PrefillArgs a, int total, int* off) {
  __shared__ int part[1024];
  const int N = a.N, per = (N + 1023) / 1024, n0 = threadIdx.x * per;
  int s = 0;
  for (int i = 0; i < per; ++i) {
    const int n = n0 + i;
    if (n < N) {
      int64_t b, t0;
      int len;
      bwdc::seq_span(a, n, b, t0, len);
      s += (len + kC - 1) / kC;
    }
  }
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < 1024; ++i) {
      const int x = part[i];
      part[i] = run;
      run += x;
    }
    off[N] = min(run, total);
  }
  __syncthreads();
  int run = part[threadIdx.x];
  for (int i = 0; i < per; ++i) {
    const int n = n0 + i;
    if (n < N) {
      int64_t b, t0;
      int len;
      bwdc::seq_span(a, n, b, t0, len);
      off[n] = min(run, total);
      run += (len + kC - 1) / kC;
    }
  }
}

// chunk indices to allocate (an upper bound with varlen); may exceed INT32_MAX
int64_t chunk_total(const PrefillArgs& a) {
  const int64_t nck = ((int64_t)a.T + kC - 1) / kC;
  return a.cu_seqlens ? nck + a.N : nck * a.N;
}

size_t rec_floats(int dk, int dv) {
  return (size_t)4 * kC * dk + (size_t)2 * kC * dv + dk + (size_t)dk * dv + kC * kC;
}
size_t st_floats(int dk, int dv) { return (size_t)2 * dk * dv + (size_t)2 * kC * dv; }
size_t off_bytes(const PrefillArgs& a) {
  return a.cu_seqlens ? (((size_t)(a.N + 1) * 4 + 255) & ~(size_t)255) : 0;
}

template <class K>
cudaError_t smem_attr(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DK, int DV, typename T>
cudaError_t run(const ChunkBwdArgs& ca, cudaStream_t s) {
  using PS = bwdc::PrepSmem<DK, DV>;
  using SS = bwdc::PassSmem<DK>;
  using GS = bwdc::GradSmem<DK, DV>;
  static_assert(bwdc::Rec<DK, DV>::SIZE == (int64_t)4 * kC * DK + 2 * kC * DV + DK + DK * DV + kC * kC, "");
  cudaError_t e;
  auto* prep = kda_bwd_prep_kernel<DK, DV, T>;
  auto* sfwd = kda_bwd_state_fwd_kernel<DK, DV, T>;
  auto* srev = kda_bwd_state_rev_kernel<DK, DV, T>;
  auto* grad = kda_bwd_grad_kernel<DK, DV, T>;
  if ((e = smem_attr(prep, PS::BYTES)) != cudaSuccess || (e = smem_attr(sfwd, SS::BYTES)) != cudaSuccess ||
      (e = smem_attr(srev, SS::BYTES)) != cudaSuccess || (e = smem_attr(grad, GS::BYTES)) != cudaSuccess)
    return e;
  const PrefillArgs& a = ca.b.f;
  const dim3 cgrid((unsigned)ca.total, (unsigned)a.H);
  const unsigned pgrid = (unsigned)((int64_t)a.N * a.H * (DV / kW));
  // with no chunks at all only the reverse pass runs (it copies d_final_state to
  // d_initial_state)
  if (ca.total > 0) {
    if (chunk_grad_tc_supported(a)) {
      if ((e = launch_chunk_prep_tc(ca, s)) != cudaSuccess) return e;
    } else {
      launch_begin(s);
      prep<<<cgrid, 256, PS::BYTES, s>>>(ca);
      if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
    }
    if (chunk_grad_tc_supported(a)) {
      if ((e = launch_chunk_pass_tc(ca, false, s)) != cudaSuccess) return e;
    } else {
      launch_begin(s);
      sfwd<<<pgrid, bwdc::kPassThreads, SS::BYTES, s>>>(ca);
      if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
    }
  }
  if (chunk_grad_tc_supported(a)) {
    if ((e = launch_chunk_pass_tc(ca, true, s)) != cudaSuccess) return e;
  } else {
    launch_begin(s);
    srev<<<pgrid, bwdc::kPassThreads, SS::BYTES, s>>>(ca);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  if (ca.total > 0) {
    if (chunk_grad_tc_supported(a)) return launch_chunk_grad_tc(ca, s);  // d_k = d_v = 128, bf16
    launch_begin(s);
    grad<<<cgrid, 256, GS::BYTES, s>>>(ca);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t chunk_backward_workspace_bytes(const PrefillArgs& a) {
  const size_t per = (size_t)a.H * (rec_floats(a.dk, a.dv) + st_floats(a.dk, a.dv)) * 4;
  const int64_t total = chunk_total(a);
  return total > INT32_MAX ? 0 : off_bytes(a) + (size_t)total * per;
}

cudaError_t launch_chunk_backward(const BackwardArgs& ba, void* ws, cudaStream_t s) {
  const PrefillArgs& a = ba.f;
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  ChunkBwdArgs ca;
  ca.b = ba;
  ca.nck = (a.T + kC - 1) / kC;
  const int64_t total = chunk_total(a);
  if (total > INT32_MAX) return cudaErrorInvalidValue;  // chunk indices are int
  ca.total = (int)total;
  char* base = static_cast<char*>(ws);
  ca.off = a.cu_seqlens ? reinterpret_cast<const int*>(base) : nullptr;
  ca.rec = reinterpret_cast<float*>(base + off_bytes(a));
  ca.st = ca.rec + (size_t)ca.total * a.H * rec_floats(a.dk, a.dv);
  cudaError_t e;
  if (a.cu_seqlens) {
    launch_begin(s);
    kda_bwd_offsets_kernel<<<1, 1024, 0, s>>>(a, ca.total, reinterpret_cast<int*>(base));
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  const bool bf = a.bf16 != 0;
#define KDA_BWDC(DK_, DV_) \
  if (a.dk == DK_ && a.dv == DV_) return bf ? run<DK_, DV_, __nv_bfloat16>(ca, s) : run<DK_, DV_, float>(ca, s);
  KDA_BWDC(128, 128)
  KDA_BWDC(128, 64)
  KDA_BWDC(64, 128)
  KDA_BWDC(64, 64)
#undef KDA_BWDC
  return cudaErrorInvalidValue;
}

}  // namespace kda
