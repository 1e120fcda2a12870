// SIMT kernels of the KDA core:
//   * kda_decode_kernel     - one decode token per (request, head), state in place;
//   * kda_recurrent_kernel  - token-recurrent prefill with the state held in
//                             registers, four tokens per pass over the state (the
//                             fp32-input path, any sequence length), also the
//                             multi-token decode step (requests as sequences, the
//                             state kept after an accepted count);
//   * kda_decode_front_kernel, kda_decode_back_kernel - the front end (short
//                             convolutions, SiLU, L2 norms) and back end (RMS
//                             norm, output gate) around kda_decode_kernel in the
//                             fused decode step;
//   * kda_backward_kernel   - reverse-mode derivative of the token recurrence;
//   * kda_seqlens_kernel    - device-side validation of cu_seqlens.
//
// The decode kernel runs the single-step recurrence in the order of
// "Kimi K3 核心算子拆解" (devpress.csdn.net) §2.3: decay every key-channel row by
// alpha_i = exp(g_i), subtract beta k (k^T S), add beta k v^T, then read out
// o = scale * S^T q ("Kimi K3 技术报告解读" (marsggbo.github.io) §3.2).  The
// correction and the write are two fused multiply-adds per element,
//   S' = fma(beta k_i, v_j, fma(-beta k_i, (k^T S)_j, S_ij)),
// so a unit key with beta = 1 reproduces v exactly in that row.  The
// token-recurrent kernel takes the same recurrence four tokens at a time in its
// unrolled form (derived above that kernel): the same values up to fp32
// rounding, with the state read twice and written once per four tokens.
//
// Thread layout of the decode and token-recurrent kernels (128 threads per
// (sequence|request, head, 64 value columns); four CTAs per SM for the decode
// step, five for the token-recurrent kernel): a 64-column
// state row slice is covered by 16 threads holding 4 consecutive columns (one
// 16-byte vector each); 8 rows are handled side by side and each thread keeps
// d_k/8 rows in registers.  (The backward kernel uses 256 threads, 16 rows side
// by side.)  Column sums over the key channels are reduced through shared
// memory.  A warp loads and stores two 256-byte row slices per instruction.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 128;  // threads of the decode and token-recurrent kernels

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ void fma4(float4& acc, float s, const float4& x) {
  acc.x = fmaf(s, x.x, acc.x);
  acc.y = fmaf(s, x.y, acc.y);
  acc.z = fmaf(s, x.z, acc.z);
  acc.w = fmaf(s, x.w, acc.w);
}

// asynchronous global -> shared copies (the token-recurrent kernel's inputs)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// S' = fma(bk, v, fma(-bk, kS, S)) element-wise
__device__ __forceinline__ float4 delta_write(float4 s, float bk, const float4& kS, const float4& v) {
  s.x = fmaf(bk, v.x, fmaf(-bk, kS.x, s.x));
  s.y = fmaf(bk, v.y, fmaf(-bk, kS.y, s.y));
  s.z = fmaf(bk, v.z, fmaf(-bk, kS.z, s.z));
  s.w = fmaf(bk, v.w, fmaf(-bk, kS.w, s.w));
  return s;
}

template <int DK, int DV, int NT = kThreads>
struct Layout {
  static constexpr int TPR = DV / 4;           // threads per state row
  static constexpr int RPP = NT / TPR;         // rows side by side
  static constexpr int R = DK / RPP;           // rows per thread
  static_assert(R * RPP == DK, "layout");
};

// Sum over the RPP row groups of per-thread partial column sums, every thread
// forming the totals of its column quad (the decode step, whose reductions hide
// behind its HBM traffic).
template <int DK, int DV, int NT = kThreads>
__device__ __forceinline__ float4 column_reduce(float4 part, float4 (*red)[DV / 4], int trow,
                                               int col4) {
  using L = Layout<DK, DV, NT>;
  red[trow][col4] = part;
  __syncthreads();
  float4 s = red[0][col4];
#pragma unroll
  for (int r = 1; r < L::RPP; ++r) {
    const float4 x = red[r][col4];
    s.x += x.x;
    s.y += x.y;
    s.z += x.z;
    s.w += x.w;
  }
  return s;
}

// The same sums in the same order, formed once per column quad: the TPR threads of
// row group 0 add the RPP partials and publish the totals in `tot` (one more
// barrier, one sixteenth of the shared-memory reads).  For the backward's token
// loop, whose reductions are not hidden behind HBM traffic.
template <int DK, int DV, int NT = kThreads>
__device__ __forceinline__ float4 column_reduce_lean(float4 part, float4 (*red)[DV / 4], float4* tot,
                                                    int trow, int col4) {
  using L = Layout<DK, DV, NT>;
  red[trow][col4] = part;
  __syncthreads();
  if (trow == 0) {
    float4 s = red[0][col4];
#pragma unroll
    for (int r = 1; r < L::RPP; ++r) {
      const float4 x = red[r][col4];
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    tot[col4] = s;
  }
  __syncthreads();
  return tot[col4];
}

// ---------------------------------------------------------------------------
// decode: one CTA per (request, head); every state element read once, written once
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kTok, 4) kda_decode_kernel(DecodeArgs a) {
  using L = Layout<DK, DV, kTok>;
  __shared__ float s_q[DK], s_k[DK], s_a[DK];
  __shared__ float4 red0[L::RPP][DV / 4];
  __shared__ float4 red1[L::RPP][DV / 4];
  const int nsl = a.dv / DV;                 // CTAs per (request, head): DV columns each
  const int col0 = (blockIdx.x % nsl) * DV;
  const int nh = blockIdx.x / nsl;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int64_t ld = a.dv;                   // state row stride
  const int tid = threadIdx.x;
  const int col4 = tid % L::TPR;
  const int trow = tid / L::TPR;

  float* S = a.state + n * a.s_sn + h * a.s_sh + col0;
  float4 s[L::R];
#pragma unroll
  for (int r = 0; r < L::R; ++r)
    s[r] = __ldcs(reinterpret_cast<const float4*>(S + (trow + L::RPP * r) * ld + 4 * col4));

  const T* qp = static_cast<const T*>(a.q.ptr) + n * a.q.sb + h * a.q.sh;
  const T* kp = static_cast<const T*>(a.k.ptr) + n * a.k.sb + h * a.k.sh;
  const float* gp = static_cast<const float*>(a.g.ptr) + n * a.g.sb + h * a.g.sh;
  const T* vp = static_cast<const T*>(a.v.ptr) + n * a.v.sb + h * a.v.sh + col0;
  const float beta = __ldg(a.beta + n * a.beta_sn + h * a.beta_sh);
  if (tid < DK) {
    s_q[tid] = to_f(qp[tid]);
    s_k[tid] = to_f(kp[tid]);
    s_a[tid] = expf(__ldg(gp + tid));
  }
  const float4 v4 = load4<T>(vp + 4 * col4);
  __syncthreads();

  float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < L::R; ++r) {
    const int i = trow + L::RPP * r;
    const float al = s_a[i];
    s[r].x *= al;
    s[r].y *= al;
    s[r].z *= al;
    s[r].w *= al;
    fma4(part, s_k[i], s[r]);
  }
  const float4 kS = column_reduce<DK, DV, kTok>(part, red0, trow, col4);

  float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < L::R; ++r) {
    const int i = trow + L::RPP * r;
    s[r] = delta_write(s[r], beta * s_k[i], kS, v4);
    __stcs(reinterpret_cast<float4*>(S + i * ld + 4 * col4), s[r]);
    fma4(po, s_q[i], s[r]);
  }
  float4 o = column_reduce<DK, DV, kTok>(po, red1, trow, col4);
  if (trow == 0) {
    o.x *= a.scale;
    o.y *= a.scale;
    o.z *= a.scale;
    o.w *= a.scale;
    store4<T>(static_cast<T*>(a.out) + n * a.out_sn + h * a.out_sh + col0 + 4 * col4, o);
  }
}

// ---------------------------------------------------------------------------
// fused decode: front end (short convolutions, SiLU, L2 norm of q and k), the
// decode step, back end (head RMSNorm, sigmoid output gate).  Three launches:
// the step itself is the plain decode kernel on fp32 inputs, at its own
// occupancy (four 64-column CTAs per SM); one kernel holding a whole head for
// the RMS norm ran at two thirds of that.  The front and back ends move a few
// hundred bytes per (request, head), the step 128 KB.

// Sum of one value per thread over the first `nthr` threads (a multiple of 32),
// returned to every thread.  `buf` holds kThreads / 32 floats; two barriers.
__device__ __forceinline__ float block_sum(float x, float* buf, int nthr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  if (lane == 0) buf[warp] = x;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < nthr / 32; ++w) s += buf[w];
  __syncthreads();
  return s;
}

// Two adjacent channels per thread in the fused decode's front and back ends (the
// host requires the conv caches to be aligned to a channel pair).
template <typename T>
struct Pair;
template <>
struct Pair<float> {
  using type = float2;
  static __device__ __forceinline__ float2 f(float2 p) { return p; }
  static __device__ __forceinline__ float2 make(float x, float y) { return make_float2(x, y); }
};
template <>
struct Pair<__nv_bfloat16> {
  using type = __nv_bfloat162;
  static __device__ __forceinline__ float2 f(__nv_bfloat162 p) { return __bfloat1622float2(p); }
  static __device__ __forceinline__ __nv_bfloat162 make(float x, float y) { return __floats2bfloat162_rn(x, y); }
};

// conv (width 4, causal, depthwise) of channels c and c + 1 over their three
// cached raw inputs and the new one, then SiLU; the cache slots move down by one
// and the raw inputs enter the newest slot (cache and x point at channel c)
template <typename T>
__device__ __forceinline__ float2 conv_silu_update2(T* cache, int64_t slot_stride, const T* x, const float* w) {
  using P = typename Pair<T>::type;
  P* c = reinterpret_cast<P*>(cache);
  const P r0 = c[0], r1 = c[slot_stride / 2], r2 = c[slot_stride], raw = *reinterpret_cast<const P*>(x);
  const float2 c0 = Pair<T>::f(r0), c1 = Pair<T>::f(r1), c2 = Pair<T>::f(r2), xv = Pair<T>::f(raw);
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w)), w1 = __ldg(reinterpret_cast<const float4*>(w + 4));
  const float y0 = w0.x * c0.x + w0.y * c1.x + w0.z * c2.x + w0.w * xv.x;
  const float y1 = w1.x * c0.y + w1.y * c1.y + w1.z * c2.y + w1.w * xv.y;
  c[0] = r1;
  c[slot_stride / 2] = r2;
  c[slot_stride] = raw;
  return make_float2(y0 / (1.f + expf(-y0)), y1 / (1.f + expf(-y1)));
}

// Front end, one CTA of max(d_k, d_v) / 2 threads per (request, head), channels
// 2t and 2t + 1 on thread t: the fp32 inputs of the step, [q^ | k^ | v^] per
// (request, head) in `x`.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__((DK > DV ? DK : DV) / 2) kda_decode_front_kernel(FusedDecodeArgs fa, float* x) {
  const DecodeArgs& a = fa.d;
  __shared__ float s_buf[kThreads / 32];
  const int nh = blockIdx.x;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int c = 2 * threadIdx.x;
  float2 qa = make_float2(0.f, 0.f), ka = make_float2(0.f, 0.f);
  if (c < DK) {
    T* cq = static_cast<T*>(fa.cq) + n * fa.cq_sn + h * fa.cq_sh + c;
    T* ck = static_cast<T*>(fa.ck) + n * fa.ck_sn + h * fa.ck_sh + c;
    qa = conv_silu_update2<T>(cq, fa.cq_ss, static_cast<const T*>(a.q.ptr) + n * a.q.sb + h * a.q.sh + c,
                              fa.wq + ((int64_t)h * DK + c) * 4);
    ka = conv_silu_update2<T>(ck, fa.ck_ss, static_cast<const T*>(a.k.ptr) + n * a.k.sb + h * a.k.sh + c,
                              fa.wk + ((int64_t)h * DK + c) * 4);
  }
  float* xo = x + (int64_t)nh * (2 * DK + DV);
  if (c < DV) {
    T* cv = static_cast<T*>(fa.cv) + n * fa.cv_sn + h * fa.cv_sh + c;
    *reinterpret_cast<float2*>(xo + 2 * DK + c) =
        conv_silu_update2<T>(cv, fa.cv_ss, static_cast<const T*>(a.v.ptr) + n * a.v.sb + h * a.v.sh + c,
                             fa.wv + ((int64_t)h * DV + c) * 4);
  }
  const float nq = sqrtf(block_sum(qa.x * qa.x + qa.y * qa.y, s_buf, DK / 2));
  const float nk = sqrtf(block_sum(ka.x * ka.x + ka.y * ka.y, s_buf, DK / 2));
  if (c < DK) {
    const float iq = 1.f / fmaxf(nq, 1e-6f), ik = 1.f / fmaxf(nk, 1e-6f);
    *reinterpret_cast<float2*>(xo + c) = make_float2(qa.x * iq, qa.y * iq);
    *reinterpret_cast<float2*>(xo + DK + c) = make_float2(ka.x * ik, ka.y * ik);
  }
}

// Back end, one CTA of d_v / 2 threads per (request, head), columns 2t and 2t + 1
// on thread t: the step's output o (fp32, already times scale) -> o / rms(o) * w *
// sigmoid(gate).
template <int DV, typename T>
__global__ void __launch_bounds__(DV / 2) kda_decode_back_kernel(FusedDecodeArgs fa, const float* o) {
  const DecodeArgs& a = fa.d;
  __shared__ float s_buf[kThreads / 32];
  const int nh = blockIdx.x;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int c = 2 * threadIdx.x;
  const float2 y = *reinterpret_cast<const float2*>(o + (int64_t)nh * DV + c);
  const float inv = rsqrtf(block_sum(y.x * y.x + y.y * y.y, s_buf, DV / 2) / DV + fa.eps);
  using P = typename Pair<T>::type;
  const float2 gl = Pair<T>::f(*reinterpret_cast<const P*>(static_cast<const T*>(fa.gate.ptr) + n * fa.gate.sb +
                                                             h * fa.gate.sh + c));
  const float2 w = fa.norm_w ? __ldg(reinterpret_cast<const float2*>(fa.norm_w + c)) : make_float2(1.f, 1.f);
  *reinterpret_cast<P*>(static_cast<T*>(a.out) + n * a.out_sn + h * a.out_sh + c) =
      Pair<T>::make(y.x * inv * w.x / (1.f + expf(-gl.x)), y.y * inv * w.y / (1.f + expf(-gl.y)));
}

// ---------------------------------------------------------------------------
// backward: one CTA per (sequence, head), all d_v columns (the gradients of q, k
// and g sum over them).  Reverse-mode derivative of the token step
//   Sb = Diag(alpha) S_prev;  delta = v - Sb^T k;  S = Sb + beta k delta^T;
//   o = scale S^T q
// run backwards with the running gradient dS (of the state after the token):
//   dS += scale q do^T;  dq = scale S do;  c = dS^T k;  ddelta = beta c;  dv = ddelta;
//   dbeta = delta . c;  dk = beta dS delta - Sb ddelta;  dSb = dS - k ddelta^T;
//   dalpha = rowsum(dSb * S_prev);  dg = dalpha * alpha;  dS <- Diag(alpha) dSb.
// The states entering each token are recomputed: a forward pass stores every
// kBwdBlock-th state, and each block is replayed into a scratch area before its
// tokens are differentiated in reverse.

// Sum of x over the TPR threads of a row group (all of them get the sum).
template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off, TPR);
  return x;
}

// One CTA per (sequence, head, DV = 32 or 64 value columns).  With two slices the
// row sums (dq, dk, dg, dbeta) are added atomically into outputs zeroed
// beforehand: two fp32 adds onto zero give the same bits in either order.  With
// four, slices 0-1 add into the outputs and slices 2-3 into a zeroed scratch
// copy, which a last kernel adds in: the result is again independent of order.
template <int DK, int DV, typename T, int NT>
__global__ void __launch_bounds__(NT, 1) kda_backward_kernel(BackwardArgs ba) {
  using L = Layout<DK, DV, NT>;
  const PrefillArgs& a = ba.f;
  __shared__ float s_q[2][DK], s_k[2][DK], s_a[2][DK];
  __shared__ float4 red0[L::RPP][DV / 4];
  __shared__ float4 red1[L::RPP][DV / 4];
  __shared__ float4 tot0[DV / 4], tot1[DV / 4];
  const int nsl = a.dv / DV;
  const bool split = nsl > 1;
  const int col0 = (blockIdx.x % nsl) * DV;
  const int nh = blockIdx.x / nsl;
  // four slices: slices 2-3 add their row sums into ba.part, so that every output
  // element gets exactly two atomic terms (the same bits in either order)
  const bool to_part = nsl == 4 && (blockIdx.x % nsl) >= 2;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int64_t ld = a.dv;  // row stride of the state and its gradients
  const int tid = threadIdx.x;
  const int col4 = tid % L::TPR;
  const int trow = tid / L::TPR;
  const int64_t blk_stride = (int64_t)DK * DV;  // workspace states hold this CTA's columns only

  int64_t b = n, t0 = 0, t1 = a.T;
  if (a.cu_seqlens) {
    b = 0;
    t0 = min(max(__ldg(a.cu_seqlens + n), 0), a.T);
    t1 = min(max(__ldg(a.cu_seqlens + n + 1), (int)t0), a.T);
  }
  const T* qb = static_cast<const T*>(a.q.ptr) + b * a.q.sb + h * a.q.sh;
  const T* kb = static_cast<const T*>(a.k.ptr) + b * a.k.sb + h * a.k.sh;
  const float* gb = static_cast<const float*>(a.g.ptr) + b * a.g.sb + h * a.g.sh;
  const T* vb = static_cast<const T*>(a.v.ptr) + b * a.v.sb + h * a.v.sh + col0;
  const float* bb = a.beta + b * a.beta_sb + h * a.beta_sh;
  const T* dob = static_cast<const T*>(ba.dout.ptr) + b * ba.dout.sb + h * ba.dout.sh + col0;
  float* ck = ba.ck + (int64_t)blockIdx.x * ba.nblk * blk_stride;
  float* scr = ba.scr + (int64_t)blockIdx.x * kBwdBlock * blk_stride;

  auto store_state = [&](float* dst, const float4 (&x)[L::R]) {
#pragma unroll
    for (int r = 0; r < L::R; ++r)
      *reinterpret_cast<float4*>(dst + (trow + L::RPP * r) * DV + 4 * col4) = x[r];
  };
  auto load_state = [&](const float* src, float4 (&x)[L::R]) {
#pragma unroll
    for (int r = 0; r < L::R; ++r)
      x[r] = *reinterpret_cast<const float4*>(src + (trow + L::RPP * r) * DV + 4 * col4);
  };
  // token t's q, k, alpha into buffer buf (threads < DK); one barrier follows
  auto stage = [&](int64_t t, int buf) {
    if (tid < DK) {
      s_q[buf][tid] = to_f(qb[t * a.q.st + tid]);
      s_k[buf][tid] = to_f(kb[t * a.k.st + tid]);
      s_a[buf][tid] = expf(__ldg(gb + t * a.g.st + tid));
    }
  };
  // one forward step of the state in registers (no read-out)
  auto forward = [&](float4 (&x)[L::R], int64_t t, int buf) {
    const float4 v4 = load4<T>(vb + t * a.v.st + 4 * col4);
    const float beta = __ldg(bb + t * a.beta_st);
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < L::R; ++r) {
      const int i = trow + L::RPP * r;
      const float al = s_a[buf][i];
      x[r].x *= al;
      x[r].y *= al;
      x[r].z *= al;
      x[r].w *= al;
      fma4(part, s_k[buf][i], x[r]);
    }
    const float4 kS = column_reduce_lean<DK, DV, NT>(part, red0, tot0, trow, col4);
#pragma unroll
    for (int r = 0; r < L::R; ++r) x[r] = delta_write(x[r], beta * s_k[buf][trow + L::RPP * r], kS, v4);
  };

  // ---- pass 1: the state entering every kBwdBlock-th token ----
  float4 S[L::R];
  if (a.s0) {
    const float* S0 = a.s0 + n * a.s0_sn + h * a.s0_sh + col0;
#pragma unroll
    for (int r = 0; r < L::R; ++r)
      S[r] = *reinterpret_cast<const float4*>(S0 + (trow + L::RPP * r) * ld + 4 * col4);
  } else {
#pragma unroll
    for (int r = 0; r < L::R; ++r) S[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int pbuf = 0;
  for (int64_t t = t0; t < t1; ++t) {
    if ((t - t0) % kBwdBlock == 0) store_state(ck + ((t - t0) / kBwdBlock) * blk_stride, S);
    stage(t, pbuf);
    __syncthreads();
    forward(S, t, pbuf);
    pbuf ^= 1;
  }

  // ---- pass 2: blocks in reverse ----
  float4 dS[L::R];
  if (ba.dsT) {
    const float* D = ba.dsT + n * ba.dsT_sn + h * ba.dsT_sh + col0;
#pragma unroll
    for (int r = 0; r < L::R; ++r)
      dS[r] = *reinterpret_cast<const float4*>(D + (trow + L::RPP * r) * ld + 4 * col4);
  } else {
#pragma unroll
    for (int r = 0; r < L::R; ++r) dS[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t nb = (t1 - t0 + kBwdBlock - 1) / kBwdBlock;
  for (int64_t blk = nb - 1; blk >= 0; --blk) {
    const int64_t ta = t0 + blk * kBwdBlock, tb = min(ta + kBwdBlock, t1);
    // replay the block: scratch[t - ta] = state entering token t (each thread reads
    // back only the elements it wrote)
    load_state(ck + blk * blk_stride, S);
    for (int64_t t = ta; t < tb; ++t) {
      store_state(scr + (t - ta) * blk_stride, S);
      stage(t, pbuf);
      __syncthreads();
      forward(S, t, pbuf);
      pbuf ^= 1;
    }
    for (int64_t t = tb - 1; t >= ta; --t) {
      stage(t, pbuf);
      const float4 v4 = load4<T>(vb + t * a.v.st + 4 * col4);
      const float4 do4 = load4<T>(dob + t * ba.dout.st + 4 * col4);
      const float beta = __ldg(bb + t * a.beta_st);
      float4 Sp[L::R];
      load_state(scr + (t - ta) * blk_stride, Sp);
      __syncthreads();
      const int buf = pbuf;
      pbuf ^= 1;
      // Sb = Diag(alpha) S_prev; delta = v - Sb^T k
      float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < L::R; ++r) {
        const int i = trow + L::RPP * r;
        const float al = s_a[buf][i];
        float4 sb = Sp[r];
        sb.x *= al;
        sb.y *= al;
        sb.z *= al;
        sb.w *= al;
        fma4(part, s_k[buf][i], sb);
      }
      const float4 kS = column_reduce_lean<DK, DV, NT>(part, red0, tot0, trow, col4);
      const float4 dl = make_float4(v4.x - kS.x, v4.y - kS.y, v4.z - kS.z, v4.w - kS.w);
      // dS += scale q do^T; dq = scale S do (S = Sb + beta k delta^T); c = dS^T k
      float dqr[L::R];
      float4 cp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < L::R; ++r) {
        const int i = trow + L::RPP * r;
        const float al = s_a[buf][i], ki = s_k[buf][i], qi = s_q[buf][i];
        const float bk = beta * ki;
        const float4 st = make_float4(fmaf(bk, dl.x, al * Sp[r].x), fmaf(bk, dl.y, al * Sp[r].y),
                                      fmaf(bk, dl.z, al * Sp[r].z), fmaf(bk, dl.w, al * Sp[r].w));
        dqr[r] = st.x * do4.x + st.y * do4.y + st.z * do4.z + st.w * do4.w;
        const float sq = a.scale * qi;
        dS[r].x = fmaf(sq, do4.x, dS[r].x);
        dS[r].y = fmaf(sq, do4.y, dS[r].y);
        dS[r].z = fmaf(sq, do4.z, dS[r].z);
        dS[r].w = fmaf(sq, do4.w, dS[r].w);
        fma4(cp, ki, dS[r]);
      }
      const float4 c = column_reduce_lean<DK, DV, NT>(cp, red1, tot1, trow, col4);
      const float4 dd = make_float4(beta * c.x, beta * c.y, beta * c.z, beta * c.w);
      // dk = beta dS delta - Sb ddelta; dSb = dS - k ddelta^T; dalpha = rowsum(dSb * S_prev)
      float dkr[L::R], dar[L::R];
#pragma unroll
      for (int r = 0; r < L::R; ++r) {
        const int i = trow + L::RPP * r;
        const float al = s_a[buf][i], ki = s_k[buf][i];
        dkr[r] = beta * (dS[r].x * dl.x + dS[r].y * dl.y + dS[r].z * dl.z + dS[r].w * dl.w) -
                 al * (Sp[r].x * dd.x + Sp[r].y * dd.y + Sp[r].z * dd.z + Sp[r].w * dd.w);
        float4 dsb = make_float4(fmaf(-ki, dd.x, dS[r].x), fmaf(-ki, dd.y, dS[r].y), fmaf(-ki, dd.z, dS[r].z),
                                 fmaf(-ki, dd.w, dS[r].w));
        dar[r] = dsb.x * Sp[r].x + dsb.y * Sp[r].y + dsb.z * Sp[r].z + dsb.w * Sp[r].w;
        dS[r] = make_float4(al * dsb.x, al * dsb.y, al * dsb.z, al * dsb.w);
      }
      // Row sums over the d_v columns of this thread's dq, dk and dg rows: a
      // reduce-scatter across the TPR lanes of the row group, each exchange
      // halving what a lane holds (the list: dq rows, dk rows, dg rows, zero
      // padding); lane l ends with the totals of items [l NV/TPR, (l+1) NV/TPR).
      {
        constexpr int NV = ((3 * L::R + L::TPR - 1) / L::TPR) * L::TPR;
        constexpr int kPer = NV / L::TPR;
        float rs[NV];
#pragma unroll
        for (int r = 0; r < L::R; ++r) {
          rs[r] = dqr[r];
          rs[L::R + r] = dkr[r];
          rs[2 * L::R + r] = dar[r];
        }
#pragma unroll
        for (int j = 3 * L::R; j < NV; ++j) rs[j] = 0.f;
#pragma unroll
        for (int st = 1; (L::TPR >> st) > 0 && st <= 5; ++st) {
          const int m = L::TPR >> st;  // partner lane offset
          const int half = NV >> st;   // items kept after this exchange
          const bool up = (col4 & m) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float send = up ? rs[i] : rs[i + half];
            const float keep = up ? rs[i + half] : rs[i];
            rs[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int j = col4 * kPer + i;
          if (j < 3 * L::R) {
            const int kind = j / L::R, rr = j - kind * L::R;  // 0: dq, 1: dk, 2: dg
            const int row = trow + L::RPP * rr;
            float* p;
            float val = rs[i];
            if (kind == 0) {
              p = ba.dq.ptr + b * ba.dq.sb + t * ba.dq.st + h * ba.dq.sh + row;
              val *= a.scale;
            } else if (kind == 1) {
              p = ba.dk.ptr + b * ba.dk.sb + t * ba.dk.st + h * ba.dk.sh + row;
            } else {
              p = ba.dg.ptr + b * ba.dg.sb + t * ba.dg.st + h * ba.dg.sh + row;
              val *= s_a[buf][row];
            }
            if (to_part) p = ba.part + ((b * a.T + t) * a.H + h) * 4 * DK + kind * DK + row;
            if (split)
              atomicAdd(p, val);
            else
              *p = val;
          }
        }
      }
      // dbeta = delta . c over the d_v columns: every row group holds the same columns,
      // so every group forms the same sum (all lanes take part in the shuffles)
      const float db = row_sum<L::TPR>(dl.x * c.x + dl.y * c.y + dl.z * c.z + dl.w * c.w);
      if (trow == 0) {
        *reinterpret_cast<float4*>(ba.dv.ptr + b * ba.dv.sb + t * ba.dv.st + h * ba.dv.sh + col0 + 4 * col4) = dd;
        if (col4 == 0) {
          float* pb = to_part ? ba.part + ((b * a.T + t) * a.H + h) * 4 * DK + 3 * DK
                              : ba.dbeta + b * ba.db_sb + t * ba.db_st + h * ba.db_sh;
          if (split)
            atomicAdd(pb, db);
          else
            *pb = db;
        }
      }
    }
  }
  if (ba.ds0) {
    float* D = ba.ds0 + n * ba.ds0_sn + h * ba.ds0_sh + col0;
#pragma unroll
    for (int r = 0; r < L::R; ++r)
      *reinterpret_cast<float4*>(D + (trow + L::RPP * r) * ld + 4 * col4) = dS[r];
  }
}

// Zero the row-sum gradients (dq, dk, dg over d_k, dbeta) of every token, strided views.
__global__ void kda_backward_zero_kernel(BackwardArgs ba) {
  const PrefillArgs& a = ba.f;
  const int64_t rows = (int64_t)a.B * a.T * a.H;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t h = r % a.H, bt = r / a.H, t = bt % a.T, b = bt / a.T;
    for (int i = threadIdx.x; i < a.dk; i += blockDim.x) {
      ba.dq.ptr[b * ba.dq.sb + t * ba.dq.st + h * ba.dq.sh + i] = 0.f;
      ba.dk.ptr[b * ba.dk.sb + t * ba.dk.st + h * ba.dk.sh + i] = 0.f;
      ba.dg.ptr[b * ba.dg.sb + t * ba.dg.st + h * ba.dg.sh + i] = 0.f;
    }
    if (threadIdx.x == 0) ba.dbeta[b * ba.db_sb + t * ba.db_st + h * ba.db_sh] = 0.f;
    if (ba.part)
      for (int i = threadIdx.x; i < 4 * a.dk; i += blockDim.x) ba.part[r * 4 * a.dk + i] = 0.f;
  }
}

// Four value-column slices: outputs += the row sums that slices 2-3 collected.
__global__ void kda_backward_merge_kernel(BackwardArgs ba) {
  const PrefillArgs& a = ba.f;
  const int64_t rows = (int64_t)a.B * a.T * a.H;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t h = r % a.H, bt = r / a.H, t = bt % a.T, b = bt / a.T;
    const float* pr = ba.part + r * 4 * a.dk;
    for (int i = threadIdx.x; i < a.dk; i += blockDim.x) {
      ba.dq.ptr[b * ba.dq.sb + t * ba.dq.st + h * ba.dq.sh + i] += pr[i];
      ba.dk.ptr[b * ba.dk.sb + t * ba.dk.st + h * ba.dk.sh + i] += pr[a.dk + i];
      ba.dg.ptr[b * ba.dg.sb + t * ba.dg.st + h * ba.dg.sh + i] += pr[2 * a.dk + i];
    }
    if (threadIdx.x == 0) ba.dbeta[b * ba.db_sb + t * ba.db_st + h * ba.db_sh] += pr[3 * a.dk];
  }
}

// ---------------------------------------------------------------------------
// token-recurrent prefill and multi-token decode: one CTA per (sequence, head, DV
// value columns), state in registers, tokens taken kNB at a time.  The state's
// columns evolve independently, so a (sequence, head) may be spread over
// a.dv / DV CTAs.
//
// A block of tokens 0 .. l (l < kNB) entering with state S is the single-step
// recurrence unrolled.  With G_t the in-block sum of g up to and including t,
//   delta_t = v_t - S^T (e^{G_t} k_t) - sum_{s<t} L_ts delta_s,
//   o_t     = scale (S^T (e^{G_t} q_t) + sum_{s<=t} M_ts delta_s),
//   S'      = e^{G_l} S + sum_s (beta_s e^{G_l - G_s} k_s) delta_s^T,
// L_ts = beta_s sum_i k_ti k_si e^{G_ti - G_si}, M_ts = beta_s sum_i q_ti k_si
// e^{G_ti - G_si} (every exponent a difference G_t - G_s with s <= t, or G_t
// itself: none exceeds 0 for g <= 0).  So the state is read twice (the 2 kNB
// column sums, one reduction) and written once per block, against three passes
// and two reductions per token one at a time.  Blocks start at the sequence start
// and end where the accepted tokens end, so the kept state is a block's result.
constexpr int kNB = 4;  // tokens per block of the token-recurrent kernel

// the pair terms of a block: index of L_ts (s < t) and of M_ts (s <= t)
__host__ __device__ constexpr int l_index(int t, int s) { return t * (t - 1) / 2 + s; }
__host__ __device__ constexpr int m_index(int t, int s) { return kNB * (kNB - 1) / 2 + t * (t + 1) / 2 + s; }
constexpr int kPairs = kNB * (kNB - 1) / 2 + kNB * (kNB + 1) / 2;  // 16
static_assert(kPairs == 16, "the pair reduction below handles 16 values");

// Warp sum of 16 values per lane, one value per lane pair out: at each level half
// of the values go to the partner lane, so lane bits 4..1 select the value index
// (8 b4 + 4 b3 + 2 b2 + b1) and both lanes of a pair return its full warp sum.
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w8[j] = (h16 ? v[8 + j] : v[j]) + __shfl_xor_sync(0xffffffffu, h16 ? v[j] : v[8 + j], 16);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w4[j] = (h8 ? w8[4 + j] : w8[j]) + __shfl_xor_sync(0xffffffffu, h8 ? w8[j] : w8[4 + j], 8);
#pragma unroll
  for (int j = 0; j < 2; ++j)
    w2[j] = (h4 ? w4[2 + j] : w4[j]) + __shfl_xor_sync(0xffffffffu, h4 ? w4[j] : w4[2 + j], 4);
  float w = (h2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? w2[0] : w2[1], 2);
  return w + __shfl_xor_sync(0xffffffffu, w, 1);
}

template <int DK, int DV, typename T, bool GATE>
__global__ void __launch_bounds__(kTok, 5) kda_recurrent_kernel(PrefillArgs a) {
  using L = Layout<DK, DV, kTok>;
  // a block's inputs as stored, [q | k | g or z | v] and beta per token, brought
  // in by 16-byte asynchronous copies one block ahead
  constexpr int kQB = DK * (int)sizeof(T);               // bytes of q, and of k
  constexpr int kGB = DK * (GATE ? (int)sizeof(T) : 4);  // bytes of g (or z)
  constexpr int kVB = DV * (int)sizeof(T);               // bytes of this CTA's v columns
  constexpr int kC = (2 * kQB + kGB + kVB) / 16;         // 16-byte pieces of a token's rows
  constexpr int kSlot = 16 * kC + 16;                    // + beta
  constexpr int kW = kTok / 32;
  __shared__ __align__(16) unsigned char raw[2][kNB][kSlot];
  __shared__ __align__(16) float kq[DK][2 * kNB];  // per channel: e^{G_t} k_t, then e^{G_t} q_t
  __shared__ __align__(16) float ke[DK][kNB];      // per channel: beta_t e^{G_l - G_t} k_t
  __shared__ float dec[DK];                        // e^{G_l}
  __shared__ float pair_w[kW][kPairs];             // per-warp channel sums of the pair terms
  __shared__ float lm[kPairs];                     // L and M, beta applied
  __shared__ __align__(16) float4 redp[kW][2][kNB][DV / 4];  // column sums per warp
  __shared__ __align__(16) float tot[2][kNB][DV];            // S^T (e^G k), S^T (e^G q)
  __shared__ __align__(16) float dl[kNB][DV];                // delta
  const int nsl = a.dv / DV;
  const int col0 = (blockIdx.x % nsl) * DV;  // first value column of this CTA
  const int nh = blockIdx.x / nsl;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int64_t ld = a.dv;                   // state row stride
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int col4 = tid % L::TPR;
  const int trow = tid / L::TPR;

  // token range of this sequence: rows of batch b = n, or the cu_seqlens slice
  int64_t b = n, t0 = 0, t1 = a.T;
  if (a.cu_seqlens) {
    b = 0;
    t0 = min(max(__ldg(a.cu_seqlens + n), 0), a.T);
    t1 = min(max(__ldg(a.cu_seqlens + n + 1), (int)t0), a.T);
  }

  float4 s[L::R];
  if (a.s0) {
    const float* S0 = a.s0 + n * a.s0_sn + h * a.s0_sh + col0;
#pragma unroll
    for (int r = 0; r < L::R; ++r)  // streaming: each state element is read once
      s[r] = __ldcs(reinterpret_cast<const float4*>(S0 + (trow + L::RPP * r) * ld + 4 * col4));
  } else {
#pragma unroll
    for (int r = 0; r < L::R; ++r) s[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // tokens whose update is kept (the rest still produce outputs)
  const int64_t keep = a.accepted ? min(max((int64_t)__ldg(a.accepted + n), (int64_t)0), t1 - t0) : t1 - t0;
  if (!a.out) t1 = t0 + keep;  // nothing to read out past the kept tokens
  const int64_t tk = t0 + keep;
  const bool has_q = a.q.ptr != nullptr;
  const bool outs = a.out != nullptr;

  const T* qb = has_q ? static_cast<const T*>(a.q.ptr) + b * a.q.sb + h * a.q.sh : nullptr;
  const T* kb = static_cast<const T*>(a.k.ptr) + b * a.k.sb + h * a.k.sh;
  // g given (fp32), or decay logits z in the input dtype with g = -5 sigmoid(A_h z)
  const unsigned char* gbase = static_cast<const unsigned char*>(a.g.ptr) +
                               (b * a.g.sb + h * a.g.sh) * (GATE ? (int64_t)sizeof(T) : (int64_t)4);
  const int64_t g_st = a.g.st * (GATE ? (int64_t)sizeof(T) : (int64_t)4);  // token stride, bytes
  const float gsc = GATE ? __ldg(a.gate_scale + h) : 0.f;
  const T* vb = static_cast<const T*>(a.v.ptr) + b * a.v.sb + h * a.v.sh + col0;
  const float* bb = a.beta + b * a.beta_sb + h * a.beta_sh;
  T* ob = outs ? static_cast<T*>(a.out) + b * a.out_sb + h * a.out_sh + col0 : nullptr;

  // blocks of kNB tokens over [t0, tk), then over [tk, t1)
  auto block_len = [&](int64_t tb) { return (int)min((int64_t)kNB, (tb < tk ? tk : t1) - tb); };
  auto fetch = [&](int64_t tb, int nb, int buf) {  // one 16-byte piece per thread and step
    for (int p = tid; p < nb * (kC + 1); p += kTok) {
      const int j = p / (kC + 1), c = p - j * (kC + 1);
      const int64_t t = tb + j;
      unsigned char* slot = raw[buf][j];
      if (c < kQB / 16) {
        if (has_q) cp_async16(slot + 16 * c, reinterpret_cast<const unsigned char*>(qb + t * a.q.st) + 16 * c);
      } else if (c < 2 * kQB / 16) {
        cp_async16(slot + 16 * c, reinterpret_cast<const unsigned char*>(kb + t * a.k.st) + 16 * c - kQB);
      } else if (c < (2 * kQB + kGB) / 16) {
        cp_async16(slot + 16 * c, gbase + t * g_st + 16 * c - 2 * kQB);
      } else if (c < kC) {
        cp_async16(slot + 16 * c, reinterpret_cast<const unsigned char*>(vb + t * a.v.st) + 16 * c - 2 * kQB - kGB);
      } else {
        cp_async4(slot + 16 * kC, bb + t * a.beta_st);
      }
    }
    cp_async_commit();
  };

  int64_t tb = t0;
  int nb = tb < t1 ? block_len(tb) : 0;
  int buf = 0;
  if (nb) fetch(tb, nb, 0);
  while (tb < t1) {
    const int64_t tn = tb + nb;
    const int nn = tn < t1 ? block_len(tn) : 0;
    cp_async_wait<0>();  // this thread's pieces of the block
    __syncthreads();     // (1) the block's inputs have landed; the previous block is done
    if (nn) fetch(tn, nn, buf ^ 1);

    // (2) per key channel: decay factors, scaled keys and queries, pair terms
    if (tid < DK) {
      const int i = tid;
      float kk[kNB], qq[kNB], G[kNB], bt[kNB];
      float gacc = 0.f;
#pragma unroll
      for (int j = 0; j < kNB; ++j) {
        kk[j] = qq[j] = bt[j] = 0.f;
        if (j < nb) {
          const unsigned char* slot = raw[buf][j];
          kk[j] = to_f(reinterpret_cast<const T*>(slot + kQB)[i]);
          if (has_q) qq[j] = to_f(reinterpret_cast<const T*>(slot)[i]);
          if constexpr (GATE)
            gacc += -5.f / (1.f + expf(-gsc * to_f(reinterpret_cast<const T*>(slot + 2 * kQB)[i])));
          else
            gacc += reinterpret_cast<const float*>(slot + 2 * kQB)[i];
          bt[j] = *reinterpret_cast<const float*>(slot + 16 * kC);
        }
        G[j] = gacc;
      }
      float4 kp, qp, kd;
      float* kpv = &kp.x;
      float* qpv = &qp.x;
      float* kdv = &kd.x;
#pragma unroll
      for (int j = 0; j < kNB; ++j) {
        const float e = __expf(G[j]);
        kpv[j] = kk[j] * e;
        qpv[j] = qq[j] * e;
        kdv[j] = bt[j] * kk[j] * __expf(gacc - G[j]);
      }
      *reinterpret_cast<float4*>(&kq[i][0]) = kp;
      *reinterpret_cast<float4*>(&kq[i][kNB]) = qp;
      *reinterpret_cast<float4*>(&ke[i][0]) = kd;
      dec[i] = __expf(gacc);
      float pv[kPairs];
#pragma unroll
      for (int t = 0; t < kNB; ++t) {
        pv[m_index(t, t)] = qq[t] * kk[t];
#pragma unroll
        for (int u = 0; u < t; ++u) {
          const float e = __expf(G[t] - G[u]);
          pv[l_index(t, u)] = kk[t] * kk[u] * e;
          pv[m_index(t, u)] = qq[t] * kk[u] * e;
        }
      }
      const float w = warp_sum16(pv, lane);
      if (!(lane & 1)) pair_w[warp][lane >> 1] = w;  // value index of lane pair lane/2
    } else if (lane < kPairs) {
      pair_w[warp][lane] = 0.f;  // warps beyond d_k channels
    }
    __syncthreads();  // (2)

    // (3) the block's column sums: S^T (e^{G_t} k_t), then S^T (e^{G_t} q_t); the two
    // row groups of a warp are added by one exchange
#pragma unroll
    for (int kind = 0; kind < 2; ++kind) {
      if (kind == 1 && !outs) break;
      float4 acc[kNB];
#pragma unroll
      for (int j = 0; j < kNB; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < L::R; ++r) {
        const float4 wv = *reinterpret_cast<const float4*>(&kq[trow + L::RPP * r][kind * kNB]);
        fma4(acc[0], wv.x, s[r]);
        fma4(acc[1], wv.y, s[r]);
        fma4(acc[2], wv.z, s[r]);
        fma4(acc[3], wv.w, s[r]);
      }
#pragma unroll
      for (int j = 0; j < kNB; ++j) {
        acc[j].x += __shfl_xor_sync(0xffffffffu, acc[j].x, 16);
        acc[j].y += __shfl_xor_sync(0xffffffffu, acc[j].y, 16);
        acc[j].z += __shfl_xor_sync(0xffffffffu, acc[j].z, 16);
        acc[j].w += __shfl_xor_sync(0xffffffffu, acc[j].w, 16);
        if ((lane >> 4) == kind) redp[warp][kind][j][col4] = acc[j];
      }
    }
    __syncthreads();  // (3)

    // (4) totals over the warps, in warp order; the pair terms times beta_s
    {
      const int kind = tid / (kNB * DV / 4), j = (tid / (DV / 4)) % kNB, c4 = tid % (DV / 4);
      static_assert(2 * kNB * (DV / 4) == kTok, "one column quad of one sum per thread");
      if (kind == 0 || outs) {
        float4 x = redp[0][kind][j][c4];
#pragma unroll
        for (int w = 1; w < kW; ++w) {
          const float4 y = redp[w][kind][j][c4];
          x.x += y.x;
          x.y += y.y;
          x.z += y.z;
          x.w += y.w;
        }
        *reinterpret_cast<float4*>(&tot[kind][j][4 * c4]) = x;
      }
      if (tid < kPairs) {
        // the pair's s: L entries first (t = 1.., s < t), then M (s <= t)
        int u = 0;
#pragma unroll
        for (int t = 0; t < kNB; ++t)
#pragma unroll
          for (int v = 0; v <= t; ++v) {
            if (v < t && l_index(t, v) == tid) u = v;
            if (m_index(t, v) == tid) u = v;
          }
        float p = pair_w[0][tid];
#pragma unroll
        for (int w = 1; w < kW; ++w) p += pair_w[w][tid];
        lm[tid] = u < nb ? p * *reinterpret_cast<const float*>(raw[buf][u] + 16 * kC) : 0.f;
      }
    }
    __syncthreads();  // (4)

    // (5) per value column: the deltas in token order, and the outputs
    if (tid < DV) {
      const int c = tid;
      float d[kNB];
#pragma unroll
      for (int t = 0; t < kNB; ++t) {
        d[t] = 0.f;
        if (t < nb) {
          float x = to_f(reinterpret_cast<const T*>(raw[buf][t] + 2 * kQB + kGB)[c]) - tot[0][t][c];
#pragma unroll
          for (int u = 0; u < t; ++u) x = fmaf(-lm[l_index(t, u)], d[u], x);
          d[t] = x;
          if (outs) {
            float o = tot[1][t][c];
#pragma unroll
            for (int u = 0; u <= t; ++u) o = fmaf(lm[m_index(t, u)], d[u], o);
            ob[(tb + t) * a.out_st + c] = from_f<T>(a.scale * o);
          }
        }
        dl[t][c] = d[t];
      }
    }
    __syncthreads();  // (5)

    // (6) S' = e^{G_l} S + sum_t (beta_t e^{G_l - G_t} k_t) delta_t^T
    {
      float4 d4[kNB];
#pragma unroll
      for (int j = 0; j < kNB; ++j) d4[j] = *reinterpret_cast<const float4*>(&dl[j][4 * col4]);
#pragma unroll
      for (int r = 0; r < L::R; ++r) {
        const int i = trow + L::RPP * r;
        const float4 e = *reinterpret_cast<const float4*>(&ke[i][0]);
        const float de = dec[i];
        float4 x = s[r];
        x.x *= de;
        x.y *= de;
        x.z *= de;
        x.w *= de;
        fma4(x, e.x, d4[0]);
        fma4(x, e.y, d4[1]);
        fma4(x, e.z, d4[2]);
        fma4(x, e.w, d4[3]);
        s[r] = x;
      }
    }
    const int64_t te = tn;  // tokens done: te - t0
    if (a.ckpt && ((te - t0) % a.ck_tokens) == 0 && (te - t0) / a.ck_tokens <= a.ck_count) {
      // prefix-cache checkpoint: the state after (te - t0) tokens of the sequence
      float* C = a.ckpt + ((int64_t)n * a.ck_count + (te - t0) / a.ck_tokens - 1) * a.ck_sr + h * a.ck_sh + col0;
#pragma unroll
      for (int r = 0; r < L::R; ++r) *reinterpret_cast<float4*>(C + (trow + L::RPP * r) * ld + 4 * col4) = s[r];
    }
    if (a.accepted && a.sT && te == tk) {  // the kept state: written once
      float* ST = a.sT + n * a.sT_sn + h * a.sT_sh + col0;
#pragma unroll
      for (int r = 0; r < L::R; ++r) __stcs(reinterpret_cast<float4*>(ST + (trow + L::RPP * r) * ld + 4 * col4), s[r]);
    }
    tb = tn;
    nb = nn;
    buf ^= 1;
  }
  if (a.sT && !a.accepted) {
    float* ST = a.sT + n * a.sT_sn + h * a.sT_sh + col0;
#pragma unroll
    for (int r = 0; r < L::R; ++r) __stcs(reinterpret_cast<float4*>(ST + (trow + L::RPP * r) * ld + 4 * col4), s[r]);
  }
}

__global__ void kda_seqlens_kernel(const int32_t* cu, int N, int T, int* err) {
  bool bad = false;
  for (int i = threadIdx.x; i <= N; i += blockDim.x) {
    const int c = cu[i];
    if (i == 0 && c != 0) bad = true;
    if (i == N && c != T) bad = true;
    if (i > 0 && c < cu[i - 1]) bad = true;
  }
  if (bad) atomicOr(err, kErrBadSeqlens);
}

template <template <int, int, typename> class K, typename Args>
cudaError_t dispatch(const Args& a, int dk, int dv, int bf16, dim3 grid, cudaStream_t st) {
  void (*fn)(Args) = nullptr;
#define KDA_CASE(DK_, DV_)                                                   \
  if (dk == DK_ && dv == DV_)                                                \
    fn = bf16 ? (void (*)(Args))K<DK_, DV_, __nv_bfloat16>::fn : K<DK_, DV_, float>::fn;
  KDA_CASE(64, 64)
  KDA_CASE(64, 128)
  KDA_CASE(128, 64)
  KDA_CASE(128, 128)
#undef KDA_CASE
  if (!fn) return cudaErrorInvalidValue;
  launch_begin(st);
  fn<<<grid, kTok, 0, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(st);
}

template <int DK, int DV, typename T>
struct DecodeK {
  static constexpr void (*fn)(DecodeArgs) = kda_decode_kernel<DK, DV, T>;
};

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  // 64 value columns per CTA, the layout of the recurrent kernel, so that a
  // multi-token call and the same tokens one step at a time round identically
  return dispatch<DecodeK>(a, a.dk, 64, a.bf16, dim3((unsigned)(a.N * a.H * (a.dv / 64))), s);
}

cudaError_t launch_recurrent_prefill(const PrefillArgs& a, cudaStream_t s) {
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  // 64 value columns per CTA (four CTAs per SM): for d_v = 128 a (sequence, head)
  // spreads over two CTAs, which keeps more state traffic in flight
  void (*fn)(PrefillArgs) = nullptr;
#define KDA_REC(DK_, G_) (a.bf16 ? kda_recurrent_kernel<DK_, 64, __nv_bfloat16, G_> : kda_recurrent_kernel<DK_, 64, float, G_>)
  if (a.dk == 128) fn = a.gate ? KDA_REC(128, true) : KDA_REC(128, false);
  if (a.dk == 64) fn = a.gate ? KDA_REC(64, true) : KDA_REC(64, false);
#undef KDA_REC
  if (!fn || (a.dv != 64 && a.dv != 128)) return cudaErrorInvalidValue;
  launch_begin(s);
  fn<<<dim3((unsigned)(a.N * a.H * (a.dv / 64))), kTok, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(s);
}

size_t decode_fused_workspace_bytes(int N, int H, int dk, int dv) {
  return (size_t)((int64_t)N * H * (2 * dk + 2 * dv) * 4);
}

cudaError_t launch_decode_fused(const FusedDecodeArgs& fa, void* ws, cudaStream_t s) {
  const DecodeArgs& a = fa.d;
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  void (*front)(FusedDecodeArgs, float*) = nullptr;
  void (*back)(FusedDecodeArgs, const float*) = nullptr;
#define KDA_FCASE(DK_, DV_)                                                                            \
  if (a.dk == DK_ && a.dv == DV_)                                                                      \
    front = a.bf16 ? kda_decode_front_kernel<DK_, DV_, __nv_bfloat16> : kda_decode_front_kernel<DK_, DV_, float>;
  KDA_FCASE(64, 64)
  KDA_FCASE(64, 128)
  KDA_FCASE(128, 64)
  KDA_FCASE(128, 128)
#undef KDA_FCASE
  if (a.dv == 64) back = a.bf16 ? kda_decode_back_kernel<64, __nv_bfloat16> : kda_decode_back_kernel<64, float>;
  if (a.dv == 128) back = a.bf16 ? kda_decode_back_kernel<128, __nv_bfloat16> : kda_decode_back_kernel<128, float>;
  if (!front || !back) return cudaErrorInvalidValue;
  const int64_t nh = (int64_t)a.N * a.H;
  const int64_t xs = 2 * a.dk + a.dv;  // [q^ | k^ | v^] per (request, head)
  float* x = static_cast<float*>(ws);
  float* o = x + nh * xs;
  cudaError_t e;
  launch_begin(s);
  front<<<dim3((unsigned)nh), (unsigned)((a.dk > a.dv ? a.dk : a.dv) / 2), 0, s>>>(fa, x);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  DecodeArgs d = a;  // the step on the fp32 front-end results, output to `o`
  d.q = Act{x, a.H * xs, 0, xs};
  d.k = Act{x + a.dk, a.H * xs, 0, xs};
  d.v = Act{x + 2 * a.dk, a.H * xs, 0, xs};
  d.bf16 = 0;
  d.out = o;
  d.out_sn = (int64_t)a.H * a.dv;
  d.out_sh = a.dv;
  if ((e = launch_decode(d, s)) != cudaSuccess) return e;
  launch_begin(s);
  back<<<dim3((unsigned)nh), (unsigned)(a.dv / 2), 0, s>>>(fa, o);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

int backward_value_slices(int N, int H, int dv) {
  const int sms = sm_count();
  // 32 value columns per CTA while the SMs hold them all (each CTA's token loop is
  // a latency chain: fewer columns, shorter steps), else 64
  const int64_t nh = (int64_t)N * H;
  return nh * (dv / 32) <= sms ? dv / 32 : (dv + 63) / 64;
}

size_t backward_workspace_bytes(int N, int H, int T, int64_t rows, int dk, int dv) {
  const int64_t nblk = ((int64_t)T + kBwdBlock - 1) / kBwdBlock;
  const int64_t part = backward_value_slices(N, H, dv) == 4 ? rows * H * 4 * dk : 0;
  return (size_t)(((int64_t)N * H * (nblk + kBwdBlock) * dk * dv + part) * 4);
}

cudaError_t launch_backward(const BackwardArgs& ba, cudaStream_t s) {
  const PrefillArgs& a = ba.f;
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  if (a.dv != 64 && a.dv != 128) return cudaErrorInvalidValue;
  const int nsl = backward_value_slices(a.N, a.H, a.dv);
  const int W = a.dv / nsl;  // value columns per CTA
  void (*fn)(BackwardArgs) = nullptr;
#define KDA_BWD(DK_, W_, NT_) \
  (a.bf16 ? kda_backward_kernel<DK_, W_, __nv_bfloat16, NT_> : kda_backward_kernel<DK_, W_, float, NT_>)
  if (a.dk == 128) fn = W == 32 ? KDA_BWD(128, 32, kTok) : KDA_BWD(128, 64, kThreads);
  if (a.dk == 64) fn = W == 32 ? KDA_BWD(64, 32, kTok) : KDA_BWD(64, 64, kThreads);
#undef KDA_BWD
  const int nt = W == 32 ? kTok : kThreads;
  if (!fn || (nsl == 4) != (ba.part != nullptr)) return cudaErrorInvalidValue;
  cudaError_t e;
  // zeroing and merging: one block per token row (grid-stride past 2^20 rows)
  const int64_t rows = (int64_t)a.B * a.T * a.H;
  const unsigned rgrid = (unsigned)(rows < (1 << 20) ? (rows > 0 ? rows : 1) : (1 << 20));
  if (nsl > 1) {  // partial row sums are added: start from zero
    launch_begin(s);
    kda_backward_zero_kernel<<<rgrid, 128, 0, s>>>(ba);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  launch_begin(s);
  fn<<<dim3((unsigned)(a.N * a.H * nsl)), nt, 0, s>>>(ba);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  if (nsl == 4) {
    launch_begin(s);
    kda_backward_merge_kernel<<<rgrid, 128, 0, s>>>(ba);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_check_seqlens(const int32_t* cu, int N, int T, int* err, cudaStream_t s) {
  launch_begin(s);
  kda_seqlens_kernel<<<1, 256, 0, s>>>(cu, N, T, err);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(s);
}

}  // namespace kda
