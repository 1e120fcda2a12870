// SIMT kernels of the KDA core:
//   * kda_decode_kernel     - one decode token per (request, head), state in place;
//   * kda_recurrent_kernel  - token-by-token prefill with the state held in
//                             registers (the fp32-input path, any sequence length),
//                             also the multi-token decode step (requests as
//                             sequences, the state kept after an accepted count);
//   * kda_seqlens_kernel    - device-side validation of cu_seqlens.
//
// Both compute kernels run the single-step recurrence in the order of
// "Kimi K3 核心算子拆解" (devpress.csdn.net) §2.3: decay every key-channel row by
// alpha_i = exp(g_i), subtract beta k (k^T S), add beta k v^T, then read out
// o = scale * S^T q ("Kimi K3 技术报告解读" (marsggbo.github.io) §3.2).  The
// correction and the write are two fused multiply-adds per element,
//   S' = fma(beta k_i, v_j, fma(-beta k_i, (k^T S)_j, S_ij)),
// so a unit key with beta = 1 reproduces v exactly in that row.
//
// Thread layout (256 threads per (sequence|request, head, 64 value columns)): a
// 64-column state row slice is covered by 16 threads holding 4 consecutive
// columns (one 16-byte vector each); 16 rows are handled side by side and each
// thread keeps d_k/16 rows in registers.  Column sums over the key channels
// (k^T S and q^T S) are reduced through shared memory in the same order in both
// compute kernels.  A warp loads and stores two 256-byte row slices per
// instruction.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

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

// S' = fma(bk, v, fma(-bk, kS, S)) element-wise
__device__ __forceinline__ float4 delta_write(float4 s, float bk, const float4& kS, const float4& v) {
  s.x = fmaf(bk, v.x, fmaf(-bk, kS.x, s.x));
  s.y = fmaf(bk, v.y, fmaf(-bk, kS.y, s.y));
  s.z = fmaf(bk, v.z, fmaf(-bk, kS.z, s.z));
  s.w = fmaf(bk, v.w, fmaf(-bk, kS.w, s.w));
  return s;
}

template <int DK, int DV>
struct Layout {
  static constexpr int TPR = DV / 4;           // threads per state row
  static constexpr int RPP = kThreads / TPR;   // rows side by side
  static constexpr int R = DK / RPP;           // rows per thread
  static_assert(R * RPP == DK, "layout");
};

// Sum over the RPP row groups of per-thread partial column sums (the same order
// in both compute kernels, so a token gives the same bits whichever kernel runs it).
template <int DK, int DV>
__device__ __forceinline__ float4 column_reduce(float4 part, float4 (*red)[DV / 4], int trow,
                                               int col4) {
  using L = Layout<DK, DV>;
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

// ---------------------------------------------------------------------------
// decode: one CTA per (request, head); every state element read once, written once
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kThreads, 3) kda_decode_kernel(DecodeArgs a) {
  using L = Layout<DK, DV>;
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
  const float4 kS = column_reduce<DK, DV>(part, red0, trow, col4);

  float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < L::R; ++r) {
    const int i = trow + L::RPP * r;
    s[r] = delta_write(s[r], beta * s_k[i], kS, v4);
    __stcs(reinterpret_cast<float4*>(S + i * ld + 4 * col4), s[r]);
    fma4(po, s_q[i], s[r]);
  }
  float4 o = column_reduce<DK, DV>(po, red1, trow, col4);
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
// decode step, back end (head RMSNorm, sigmoid output gate).  One CTA per
// (request, head) with all d_v columns, since the RMS norm spans them.

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

// conv (width 4, causal, depthwise) of channel c, then SiLU; the cache slots
// move down by one and the raw input enters the newest slot.
template <typename T>
__device__ __forceinline__ float conv_silu_update(T* cache, int64_t slot_stride, const T* x, const float* w) {
  const float c0 = to_f(cache[0]), c1 = to_f(cache[slot_stride]), c2 = to_f(cache[2 * slot_stride]);
  const T raw = *x;
  const float4 wv = __ldg(reinterpret_cast<const float4*>(w));
  const float y = wv.x * c0 + wv.y * c1 + wv.z * c2 + wv.w * to_f(raw);
  cache[0] = cache[slot_stride];
  cache[slot_stride] = cache[2 * slot_stride];
  cache[2 * slot_stride] = raw;
  return y / (1.f + expf(-y));
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kThreads, 2) kda_decode_fused_kernel(FusedDecodeArgs fa) {
  using L = Layout<DK, DV>;
  const DecodeArgs& a = fa.d;
  __shared__ float s_q[DK], s_k[DK], s_a[DK], s_v[DV], s_buf[kThreads / 32];
  __shared__ float4 red0[L::RPP][DV / 4];
  __shared__ float4 red1[L::RPP][DV / 4];
  const int n = blockIdx.x / a.H;
  const int h = blockIdx.x - n * a.H;
  const int tid = threadIdx.x;
  const int col4 = tid % L::TPR;
  const int trow = tid / L::TPR;

  float* S = a.state + n * a.s_sn + h * a.s_sh;
  float4 s[L::R];
#pragma unroll
  for (int r = 0; r < L::R; ++r)  // issued first: the front end runs while the state arrives
    s[r] = __ldcs(reinterpret_cast<const float4*>(S + (trow + L::RPP * r) * DV + 4 * col4));

  // ---- front end ----
  float qa = 0.f, ka = 0.f;
  if (tid < DK) {
    T* cq = static_cast<T*>(fa.cq) + n * fa.cq_sn + h * fa.cq_sh + tid;
    T* ck = static_cast<T*>(fa.ck) + n * fa.ck_sn + h * fa.ck_sh + tid;
    qa = conv_silu_update<T>(cq, fa.cq_ss, static_cast<const T*>(a.q.ptr) + n * a.q.sb + h * a.q.sh + tid,
                             fa.wq + ((int64_t)h * DK + tid) * 4);
    ka = conv_silu_update<T>(ck, fa.ck_ss, static_cast<const T*>(a.k.ptr) + n * a.k.sb + h * a.k.sh + tid,
                             fa.wk + ((int64_t)h * DK + tid) * 4);
    s_a[tid] = expf(__ldg(static_cast<const float*>(a.g.ptr) + n * a.g.sb + h * a.g.sh + tid));
  }
  if (tid < DV) {
    T* cv = static_cast<T*>(fa.cv) + n * fa.cv_sn + h * fa.cv_sh + tid;
    s_v[tid] = conv_silu_update<T>(cv, fa.cv_ss, static_cast<const T*>(a.v.ptr) + n * a.v.sb + h * a.v.sh + tid,
                                   fa.wv + ((int64_t)h * DV + tid) * 4);
  }
  const float nq = sqrtf(block_sum(qa * qa, s_buf, DK));
  const float nk = sqrtf(block_sum(ka * ka, s_buf, DK));
  if (tid < DK) {
    s_q[tid] = qa / fmaxf(nq, 1e-6f);
    s_k[tid] = ka / fmaxf(nk, 1e-6f);
  }
  const float beta = __ldg(a.beta + n * a.beta_sn + h * a.beta_sh);
  __syncthreads();
  const float4 v4 = *reinterpret_cast<const float4*>(s_v + 4 * col4);

  // ---- the decode step ----
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
  const float4 kS = column_reduce<DK, DV>(part, red0, trow, col4);
  float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < L::R; ++r) {
    const int i = trow + L::RPP * r;
    s[r] = delta_write(s[r], beta * s_k[i], kS, v4);
    __stcs(reinterpret_cast<float4*>(S + i * DV + 4 * col4), s[r]);
    fma4(po, s_q[i], s[r]);
  }
  float4 o = column_reduce<DK, DV>(po, red1, trow, col4);

  // ---- back end: the threads of row group 0 hold the d_v outputs ----
  if (trow == 0) {
    o.x *= a.scale;
    o.y *= a.scale;
    o.z *= a.scale;
    o.w *= a.scale;
    float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
    // row group 0 is lanes 0 .. TPR-1 of warp 0: only those take part
    constexpr unsigned kMask = L::TPR >= 32 ? 0xffffffffu : ((1u << L::TPR) - 1u);
#pragma unroll
    for (int off = L::TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(kMask, ss, off, L::TPR);
    const float inv = rsqrtf(ss / DV + fa.eps);
    const float4 gl = load4<T>(static_cast<const T*>(fa.gate.ptr) + n * fa.gate.sb + h * fa.gate.sh + 4 * col4);
    const float4 wn = fa.norm_w ? __ldg(reinterpret_cast<const float4*>(fa.norm_w + 4 * col4))
                                : make_float4(1.f, 1.f, 1.f, 1.f);
    o.x = o.x * inv * wn.x / (1.f + expf(-gl.x));
    o.y = o.y * inv * wn.y / (1.f + expf(-gl.y));
    o.z = o.z * inv * wn.z / (1.f + expf(-gl.z));
    o.w = o.w * inv * wn.w / (1.f + expf(-gl.w));
    store4<T>(static_cast<T*>(a.out) + n * a.out_sn + h * a.out_sh + 4 * col4, o);
  }
}

// ---------------------------------------------------------------------------
// token-by-token prefill: one CTA per (sequence, head, DV value columns), state in
// registers.  The state's columns evolve independently, so a (sequence, head)
// may be spread over a.dv / DV CTAs.
template <int DK, int DV, typename T, bool GATE>
__global__ void __launch_bounds__(kThreads, 3) kda_recurrent_kernel(PrefillArgs a) {
  using L = Layout<DK, DV>;
  __shared__ float s_q[2][DK], s_k[2][DK], s_a[2][DK];
  __shared__ float4 red0[L::RPP][DV / 4];
  __shared__ float4 red1[L::RPP][DV / 4];
  const int nsl = a.dv / DV;
  const int col0 = (blockIdx.x % nsl) * DV;  // first value column of this CTA
  const int nh = blockIdx.x / nsl;
  const int n = nh / a.H;
  const int h = nh - n * a.H;
  const int64_t ld = a.dv;                   // state row stride
  const int tid = threadIdx.x;
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
  const bool has_q = a.q.ptr != nullptr;

  const T* qb = has_q ? static_cast<const T*>(a.q.ptr) + b * a.q.sb + h * a.q.sh : nullptr;
  const T* kb = static_cast<const T*>(a.k.ptr) + b * a.k.sb + h * a.k.sh;
  // per-token decay factors alpha = e^g: g given (fp32), or g = -5 sigmoid(A_h z)
  // from decay logits z in the input dtype
  const float* gb = static_cast<const float*>(a.g.ptr) + b * a.g.sb + h * a.g.sh;
  const T* zb = static_cast<const T*>(a.g.ptr) + b * a.g.sb + h * a.g.sh;
  const float gsc = GATE ? __ldg(a.gate_scale + h) : 0.f;
  auto alpha = [&](int64_t t) {
    if constexpr (GATE) return expf(-5.f / (1.f + expf(-gsc * to_f(zb[t * a.g.st + tid]))));
    else return expf(__ldg(gb + t * a.g.st + tid));
  };
  const T* vb = static_cast<const T*>(a.v.ptr) + b * a.v.sb + h * a.v.sh + col0;
  const float* bb = a.beta + b * a.beta_sb + h * a.beta_sh;
  T* ob = a.out ? static_cast<T*>(a.out) + b * a.out_sb + h * a.out_sh + col0 : nullptr;

  // stage token t0 into buffer 0
  float pq = 0.f, pk = 0.f, pa = 0.f, pb = 0.f;
  float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (t0 < t1) {
    if (tid < DK) {
      pq = has_q ? to_f(qb[t0 * a.q.st + tid]) : 0.f;
      pk = to_f(kb[t0 * a.k.st + tid]);
      pa = alpha(t0);
    }
    pv = load4<T>(vb + t0 * a.v.st + 4 * col4);
    pb = __ldg(bb + t0 * a.beta_st);
  }
  for (int64_t t = t0; t < t1; ++t) {
    const int buf = (int)((t - t0) & 1);
    if (tid < DK) {
      s_q[buf][tid] = pq;
      s_k[buf][tid] = pk;
      s_a[buf][tid] = pa;
    }
    const float4 v4 = pv;
    const float beta = pb;
    if (t + 1 < t1) {  // prefetch the next token while this one computes
      if (tid < DK) {
        pq = has_q ? to_f(qb[(t + 1) * a.q.st + tid]) : 0.f;
        pk = to_f(kb[(t + 1) * a.k.st + tid]);
        pa = alpha(t + 1);
      }
      pv = load4<T>(vb + (t + 1) * a.v.st + 4 * col4);
      pb = __ldg(bb + (t + 1) * a.beta_st);
    }
    __syncthreads();
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < L::R; ++r) {
      const int i = trow + L::RPP * r;
      const float al = s_a[buf][i];
      s[r].x *= al;
      s[r].y *= al;
      s[r].z *= al;
      s[r].w *= al;
      fma4(part, s_k[buf][i], s[r]);
    }
    const float4 kS = column_reduce<DK, DV>(part, red0, trow, col4);
    float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < L::R; ++r) {
      const int i = trow + L::RPP * r;
      s[r] = delta_write(s[r], beta * s_k[buf][i], kS, v4);
      fma4(po, s_q[buf][i], s[r]);
    }
    if (a.ckpt && ((t - t0 + 1) % a.ck_tokens) == 0 && (t - t0 + 1) / a.ck_tokens <= a.ck_count) {
      // prefix-cache checkpoint: the state after (t - t0 + 1) tokens of the sequence
      float* C = a.ckpt + ((int64_t)n * a.ck_count + (t - t0 + 1) / a.ck_tokens - 1) * a.ck_sr + h * a.ck_sh + col0;
#pragma unroll
      for (int r = 0; r < L::R; ++r) *reinterpret_cast<float4*>(C + (trow + L::RPP * r) * ld + 4 * col4) = s[r];
    }
    if (a.accepted && a.sT && t == t0 + keep - 1) {  // the kept state: written once
      float* ST = a.sT + n * a.sT_sn + h * a.sT_sh + col0;
#pragma unroll
      for (int r = 0; r < L::R; ++r) __stcs(reinterpret_cast<float4*>(ST + (trow + L::RPP * r) * ld + 4 * col4), s[r]);
    }
    if (a.out) {
      float4 o = column_reduce<DK, DV>(po, red1, trow, col4);
      if (trow == 0) {
        o.x *= a.scale;
        o.y *= a.scale;
        o.z *= a.scale;
        o.w *= a.scale;
        store4<T>(ob + t * a.out_st + 4 * col4, o);
      }
    }
    // red0/red1 are rewritten next token only after that token's first barrier,
    // which every thread reaches after finishing its reads of this token.
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
  fn<<<grid, kThreads, 0, st>>>(a);
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
  // 64 value columns per CTA (three CTAs per SM): for d_v = 128 a (sequence, head)
  // spreads over two CTAs, which keeps more state traffic in flight
  void (*fn)(PrefillArgs) = nullptr;
#define KDA_REC(DK_, G_) (a.bf16 ? kda_recurrent_kernel<DK_, 64, __nv_bfloat16, G_> : kda_recurrent_kernel<DK_, 64, float, G_>)
  if (a.dk == 128) fn = a.gate ? KDA_REC(128, true) : KDA_REC(128, false);
  if (a.dk == 64) fn = a.gate ? KDA_REC(64, true) : KDA_REC(64, false);
#undef KDA_REC
  if (!fn || (a.dv != 64 && a.dv != 128)) return cudaErrorInvalidValue;
  launch_begin(s);
  fn<<<dim3((unsigned)(a.N * a.H * (a.dv / 64))), kThreads, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(s);
}

cudaError_t launch_decode_fused(const FusedDecodeArgs& fa, cudaStream_t s) {
  const DecodeArgs& a = fa.d;
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  void (*fn)(FusedDecodeArgs) = nullptr;
#define KDA_FCASE(DK_, DV_)                                                                     \
  if (a.dk == DK_ && a.dv == DV_)                                                               \
    fn = a.bf16 ? kda_decode_fused_kernel<DK_, DV_, __nv_bfloat16> : kda_decode_fused_kernel<DK_, DV_, float>;
  KDA_FCASE(64, 64)
  KDA_FCASE(64, 128)
  KDA_FCASE(128, 64)
  KDA_FCASE(128, 128)
#undef KDA_FCASE
  if (!fn) return cudaErrorInvalidValue;
  launch_begin(s);
  fn<<<dim3((unsigned)(a.N * a.H)), kThreads, 0, s>>>(fa);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(s);
}

cudaError_t launch_check_seqlens(const int32_t* cu, int N, int T, int* err, cudaStream_t s) {
  launch_begin(s);
  kda_seqlens_kernel<<<1, 256, 0, s>>>(cu, N, T, err);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_end(s);
}

}  // namespace kda
