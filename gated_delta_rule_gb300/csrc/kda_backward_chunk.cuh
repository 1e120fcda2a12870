// Chunked backward of the KDA core: kernel bodies.
//
// The forward is the chunked form of "尝试对Kimi KDA的数学推导&算子实现分析"
// (hjcheng0602.cn/blog/kdd): per chunk of C = 64 tokens with G the cumulative
// log-decay from the chunk start (eq. 9), K+ = K e^G, K- = K e^-G, Q+ = Q e^G,
// K_end = K e^{G_C - G} (eqs. 15-16, 64-66), L = StrictTril(diag(beta) K+ K-^T),
// T = (I + L)^-1 (eqs. 51-52), U = T diag(beta) (V - K+ S), O = scale (Q+ S +
// Tril(Q+ K-^T) U) (eqs. 36, 63) and S' = Diag(e^{G_C}) S + K_end^T U (eq. 66).
// The pages derive no backward; these kernels run the exact reverse-mode
// derivative of those equations, split into four launches:
//
//   prep    (chunk-parallel)  the state-independent chunk matrices: A = K+ K-^T,
//           T, W = T diag(beta) K+, U_bar = T diag(beta) V, and for the reverse
//           pass W_y = T^T K_end, V_y = scale T^T A_Q^T dO, Z_q = scale Q+^T dO
//   forward (per sequence, head, 32 value columns; sequential over chunks)
//           S_c for every chunk and U = U_bar - W S
//   reverse (same split, chunks in reverse) X_c, the gradient of the state leaving
//           chunk c: dY = V_y + W_y X (dv = diag(beta) dY), then
//           X <- Diag(e^{G_C}) X + Z_q - (diag(beta) K+)^T dY
//   grad    (chunk-parallel)  dq, dk, dg, dbeta of the chunk from S_c, X_c, U, dY
//
// Exponents: with g in [-5, 0] every factor e^{G_i - G_j} (j <= i) is formed as a
// product of two factors referred to the start r_J or the end c_J of a 16-token
// sub-block, each within e^{+-80}, so nothing overflows in fp32.
//
// Each body is written for `NT` threads with KB_SYNC() as its only barrier, so
// that the same source can be stepped on a host with one thread per CUDA thread.
#pragma once

#include <stdint.h>

#include "kda_internal.h"

#if defined(__CUDACC__)
#include <cuda_bf16.h>
#define KB_HD __device__ __forceinline__
#define KB_SYNC() __syncthreads()
#define KB_EXP(x) __expf(x)
#else
#include <cmath>
#include <cstring>
#define KB_HD inline
#ifndef KB_SYNC
#error "host builds define KB_SYNC()"
#endif
#define KB_EXP(x) std::exp(x)
#endif

namespace kda {
namespace bwdc {

constexpr int kC = 64;   // chunk rows
constexpr int kSB = 16;  // sub-block rows (exponent reference blocks)
constexpr int kW = 32;   // value columns per sequential CTA and per gradient-kernel slice

// Per (chunk index, head) records, fp32, offsets in floats (all multiples of 4).
template <int DK, int DV>
struct Rec {
  static constexpr int64_t W = 0;               // [64][DK]  T diag(beta) K+
  static constexpr int64_t KE = W + kC * DK;    // [64][DK]  K_end
  static constexpr int64_t UB = KE + kC * DK;   // [64][DV]  T diag(beta) V
  static constexpr int64_t EGC = UB + kC * DV;  // [DK]      e^{G_C}
  static constexpr int64_t WY = EGC + DK;       // [64][DK]  T^T K_end
  static constexpr int64_t KB = WY + kC * DK;   // [64][DK]  diag(beta) K+
  static constexpr int64_t VY = KB + kC * DK;   // [64][DV]  scale T^T A_Q^T dO
  static constexpr int64_t ZQ = VY + kC * DV;   // [DK][DV]  scale Q+^T dO
  static constexpr int64_t A = ZQ + DK * DV;    // [64][64]  strictly lower K+ K-^T
  static constexpr int64_t SIZE = A + kC * kC;
  // states and per-chunk results of the two sequential passes
  static constexpr int64_t S = 0;                // [DK][DV] state entering the chunk
  static constexpr int64_t X = S + DK * DV;      // [DK][DV] gradient of the state leaving it
  static constexpr int64_t U = X + DK * DV;      // [64][DV]
  static constexpr int64_t DY = U + kC * DV;     // [64][DV] T^T dU
  static constexpr int64_t SSIZE = DY + kC * DV;
};

struct ChunkBwdArgs {
  BackwardArgs b;  // inputs and gradients (b.ck, b.scr, b.part unused)
  const int* off;  // varlen: first chunk index of each sequence [N + 1]; null for fixed length
  int nck;         // chunks per sequence (fixed length)
  int total;       // chunk indices allocated
  float* rec;      // [total][H][Rec::SIZE]
  float* st;       // [total][H][Rec::SSIZE]
};

// 16-byte copy global -> shared that lands by the next cp_wait_all()
KB_HD void cp16(float* dst, const float* src) {
#if defined(__CUDACC__)
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
#else
  std::memcpy(dst, src, 16);
#endif
}
KB_HD void cp_commit() {
#if defined(__CUDACC__)
  asm volatile("cp.async.commit_group;\n" ::: "memory");
#endif
}
KB_HD void cp_wait_all() {
#if defined(__CUDACC__)
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
#endif
}

KB_HD float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// four consecutive elements as fp32 (8-byte aligned for bf16, 16-byte for fp32)
template <typename T>
KB_HD float4 ld4t(const T* p);
template <>
KB_HD float4 ld4t<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
#if defined(__CUDACC__)
template <>
KB_HD float4 ld4t<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xffff0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xffff0000u);
  return r;
}
#endif
KB_HD void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
KB_HD void fma4(float4& acc, float s, const float4& x) {
  acc.x += s * x.x;
  acc.y += s * x.y;
  acc.z += s * x.z;
  acc.w += s * x.w;
}
KB_HD float4 zero4() {
  float4 z;
  z.x = z.y = z.z = z.w = 0.f;
  return z;
}
KB_HD float& comp(float4& v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }
KB_HD float comp(const float4& v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }

// Where a chunk index falls: sequence n, chunk c of it, its first token row and
// its number of valid rows.
struct ChunkLoc {
  int n, c, rows;
  int64_t b, t;  // batch row and first token
};

// Token range of sequence n, clamped as the forward kernels clamp it.
KB_HD void seq_span(const PrefillArgs& a, int n, int64_t& b, int64_t& t0, int& len) {
  b = n;
  t0 = 0;
  len = a.T;
  if (a.cu_seqlens) {
    int c0 = a.cu_seqlens[n], c1 = a.cu_seqlens[n + 1];
    c0 = c0 < 0 ? 0 : (c0 > a.T ? a.T : c0);
    c1 = c1 < c0 ? c0 : (c1 > a.T ? a.T : c1);
    b = 0;
    t0 = c0;
    len = c1 - c0;
  }
}

KB_HD int first_chunk(const ChunkBwdArgs& a, int n) { return a.off ? a.off[n] : n * a.nck; }
KB_HD int num_chunks(const ChunkBwdArgs& a, int n) {
  return a.off ? a.off[n + 1] - a.off[n] : a.nck;
}

// false when chunk index f belongs to no sequence (varlen upper bound)
KB_HD bool locate(const ChunkBwdArgs& a, int f, ChunkLoc& L) {
  const PrefillArgs& p = a.b.f;
  int n;
  if (a.off) {
    if (f >= a.off[p.N]) return false;
    int lo = 0, hi = p.N - 1;  // last n with off[n] <= f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.off[mid] <= f) lo = mid;
      else hi = mid - 1;
    }
    n = lo;
  } else {
    n = f / a.nck;
  }
  int64_t b, t0;
  int len;
  seq_span(p, n, b, t0, len);
  L.n = n;
  L.c = f - first_chunk(a, n);
  L.b = b;
  L.t = t0 + (int64_t)L.c * kC;
  const int rem = len - L.c * kC;
  L.rows = rem < kC ? rem : kC;
  return L.rows > 0;
}

// A [64][D] row tile of an input with row stride `st` (zero past `rows`), as the
// 4-vectors idx = tid + u NT (row idx / (D / 4), columns 4 (idx % (D / 4)) ..): all
// loads are issued before any is used.
template <int D, int NT, typename T>
KB_HD void load_rows(float4 (&v)[kC * D / 4 / NT], const T* base, int64_t st, int rows, int tid) {
  static_assert((kC * D / 4) % NT == 0, "whole vectors per thread");
#pragma unroll
  for (int u = 0; u < kC * D / 4 / NT; ++u) {
    const int idx = tid + u * NT, i = idx / (D / 4), p = idx - i * (D / 4);
    v[u] = i < rows ? ld4t<T>(base + (int64_t)i * st + 4 * p) : zero4();
  }
}

// acc[r][c4] += sum_{j in [j0, j1)} L[4 rg + r][j] * rhs[j][4 cg + 64 c4 ..], for a
// thread holding rows 4 rg .. 4 rg + 3 and columns {4 cg + 64 c4 .. + 3} of a [64][D]
// result; L row-major with pitch lp, j0 and j1 multiples of 4.
template <int D>
KB_HD void mm64_rows(float4 (&acc)[4][D / 64], const float* L, int lp, const float* rhs, int rp, int j0,
                     int j1, int rg, int cg) {
  for (int j = j0; j < j1; j += 4) {
    float4 l[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) l[r] = ld4(L + (4 * rg + r) * lp + j);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float4 bv[D / 64];
#pragma unroll
      for (int c4 = 0; c4 < D / 64; ++c4) bv[c4] = ld4(rhs + (j + jj) * rp + 4 * cg + 64 * c4);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c4 = 0; c4 < D / 64; ++c4) fma4(acc[r][c4], comp(l[r], jj), bv[c4]);
    }
  }
}

// The same with L stored transposed: the left factor at (row 4 rg + r, j) is L[j][4 rg + r].
template <int D>
KB_HD void mm64_cols(float4 (&acc)[4][D / 64], const float* L, int lp, const float* rhs, int rp, int j0,
                     int j1, int rg, int cg) {
  for (int j = j0; j < j1; ++j) {
    const float4 l = ld4(L + j * lp + 4 * rg);
    float4 bv[D / 64];
#pragma unroll
    for (int c4 = 0; c4 < D / 64; ++c4) bv[c4] = ld4(rhs + j * rp + 4 * cg + 64 * c4);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c4 = 0; c4 < D / 64; ++c4) fma4(acc[r][c4], comp(l, r), bv[c4]);
  }
}

template <int D>
KB_HD void zero_acc(float4 (&acc)[4][D / 64]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c4 = 0; c4 < D / 64; ++c4) acc[r][c4] = zero4();
}

// stores a thread's [4][D / 64] float4 tile into a row-major [64][D] array
template <int D>
KB_HD void store64(float* dst, int pitch, const float4 (&acc)[4][D / 64], int rg, int cg) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c4 = 0; c4 < D / 64; ++c4) st4(dst + (int64_t)(4 * rg + r) * pitch + 4 * cg + 64 * c4, acc[r][c4]);
}

// ---------------------------------------------------------------------------
// prep: one CTA of 256 threads per (chunk index, head)
template <int DK, int DV>
struct PrepSmem {
  static constexpr int PM = (DK > DV ? DK : DV) + 4;  // pitch of the four [64][*] buffers
  static constexpr int PA = kC + 4;                   // pitch of the [64][64] matrices
  static constexpr int B0 = 0, B1 = B0 + kC * PM, B2 = B1 + kC * PM, B3 = B2 + kC * PM;
  static constexpr int A = B3 + kC * PM, AQ = A + kC * PA, TM = AQ + kC * PA;
  static constexpr int TAU = TM + kC * PA;  // [10][DK]: e^{r_I - r_J}, J <= I, at I (I + 1) / 2 + J
  static constexpr int RR = TAU + 10 * DK;  // [5][DK]: r_0 .. r_3 (log-decay before each sub-block), G_C
  static constexpr int BETA = RR + 5 * DK;  // [64]
  static constexpr int FLOATS = BETA + kC;
  static constexpr int BYTES = FLOATS * 4;
};

// T = (I + diag(beta) A)^-1 for a strictly lower triangular [64][64] A (row pitch pa):
// the diagonal 16 x 16 blocks by substitution, one column per thread, then block rows
// 1..3 from T_IJ = -T_II sum_K L_IK T_KJ with L = diag(beta) A.  sT (pitch pa) must be
// zero above the diagonal blocks on entry; B0 is a [16][pb] scratch.
template <int NT>
KB_HD void invert_lower(const float* sA, float* sT, const float* sb, float* B0, int pa, int pb, int tid) {
  if (tid < kC) {
    // right-looking substitution down column m of its diagonal block: s[ii] gathers
    // sum_{jj < ii} A[i][base + jj] t[jj] as the t[jj] become known
    const int base = (tid / kSB) * kSB, m = tid % kSB, col = base + m;
    float sacc[kSB], tc[kSB];
#pragma unroll
    for (int ii = 0; ii < kSB; ++ii) sacc[ii] = 0.f;
#pragma unroll
    for (int jj = 0; jj < kSB; ++jj) {
      tc[jj] = jj < m ? 0.f : jj == m ? 1.f : -sb[base + jj] * sacc[jj];
      sT[(base + jj) * pa + col] = tc[jj];
#pragma unroll
      for (int ii = jj + 1; ii < kSB; ++ii) sacc[ii] += sA[(base + ii) * pa + base + jj] * tc[jj];
    }
  }
  KB_SYNC();
  for (int I = 1; I < 4; ++I) {
    const int w = kSB * I;  // columns left of the diagonal block
    // (L T)[i][m] = beta_i sum_{kk in [16 (m / 16), w)} A[i][kk] T[kk][m]: the range is
    // a multiple of 16 long, summed in four interleaved parts
    for (int idx = tid; idx < kSB * w; idx += NT) {
      const int ii = idx / w, m = idx - ii * w, i = w + ii;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      for (int kk = (m / kSB) * kSB; kk < w; kk += 4) {
        s0 += sA[i * pa + kk] * sT[kk * pa + m];
        s1 += sA[i * pa + kk + 1] * sT[(kk + 1) * pa + m];
        s2 += sA[i * pa + kk + 2] * sT[(kk + 2) * pa + m];
        s3 += sA[i * pa + kk + 3] * sT[(kk + 3) * pa + m];
      }
      B0[ii * pb + m] = sb[i] * ((s0 + s1) + (s2 + s3));
    }
    KB_SYNC();
    // T[i][m] = -sum_kk T_II[ii][kk] (L T)[kk][m]; T_II is zero above its diagonal
    for (int idx = tid; idx < kSB * w; idx += NT) {
      const int ii = idx / w, m = idx - ii * w, i = w + ii;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int kk = 0; kk < kSB; kk += 4) {
        s0 += sT[i * pa + w + kk] * B0[kk * pb + m];
        s1 += sT[i * pa + w + kk + 1] * B0[(kk + 1) * pb + m];
        s2 += sT[i * pa + w + kk + 2] * B0[(kk + 2) * pb + m];
        s3 += sT[i * pa + w + kk + 3] * B0[(kk + 3) * pb + m];
      }
      sT[i * pa + m] = -((s0 + s1) + (s2 + s3));
    }
    KB_SYNC();
  }
}

template <int DK, int DV, typename T>
KB_HD void prep_body(const ChunkBwdArgs& ca, float* sm, int f, int h, int tid) {
  constexpr int NT = 256;
  using SM = PrepSmem<DK, DV>;
  using R = Rec<DK, DV>;
  constexpr int PM = SM::PM, PA = SM::PA;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  ChunkLoc L;
  if (!locate(ca, f, L)) return;  // uniform across the CTA
  float* rec = ca.rec + ((int64_t)f * a.H + h) * R::SIZE;
  const T* qb = static_cast<const T*>(a.q.ptr) + L.b * a.q.sb + L.t * a.q.st + (int64_t)h * a.q.sh;
  const T* kb = static_cast<const T*>(a.k.ptr) + L.b * a.k.sb + L.t * a.k.st + (int64_t)h * a.k.sh;
  const T* vb = static_cast<const T*>(a.v.ptr) + L.b * a.v.sb + L.t * a.v.st + (int64_t)h * a.v.sh;
  const T* ob = static_cast<const T*>(ba.dout.ptr) + L.b * ba.dout.sb + L.t * ba.dout.st + (int64_t)h * ba.dout.sh;
  const float* gb = static_cast<const float*>(a.g.ptr) + L.b * a.g.sb + L.t * a.g.st + (int64_t)h * a.g.sh;
  const float* bb = a.beta + L.b * a.beta_sb + L.t * a.beta_st + (int64_t)h * a.beta_sh;
  float* B0 = sm + SM::B0;
  float* B1 = sm + SM::B1;
  float* B2 = sm + SM::B2;
  float* B3 = sm + SM::B3;
  float* sA = sm + SM::A;
  float* sAQ = sm + SM::AQ;
  float* sT = sm + SM::TM;
  float* tau = sm + SM::TAU;
  float* rr = sm + SM::RR;
  float* sb = sm + SM::BETA;
  const int rows = L.rows;
  const float scale = a.scale;

  constexpr int NK = kC * DK / 4 / NT, NV = kC * DV / 4 / NT;  // 4-vectors per thread
  // 1. log-decays (zero past the last row) and beta; then per-channel cumulative sums
  {
    float4 gv[NK];
    load_rows<DK, NT, float>(gv, gb, a.g.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4);
      st4(B0 + i * PM + 4 * p, gv[u]);
    }
  }
  for (int i = tid; i < kC; i += NT) sb[i] = i < rows ? bb[(int64_t)i * a.beta_st] : 0.f;
  KB_SYNC();
  for (int d = tid; d < DK; d += NT) {
    float run = 0.f;
    rr[d] = 0.f;
    for (int i = 0; i < kC; ++i) {
      run += B0[i * PM + d];
      B0[i * PM + d] = run;
      if ((i & (kSB - 1)) == kSB - 1) rr[((i + 1) / kSB) * DK + d] = run;  // r_1..r_3, then G_C at [4]
    }
  }
  KB_SYNC();
  // 2. operands referred to the sub-block start: k e^{G - r}, k e^{r - G}, q e^{G - r}
  {
    float4 kv[NK], qv[NK];
    load_rows<DK, NT, T>(kv, kb, a.k.st, rows, tid);
    load_rows<DK, NT, T>(qv, qb, a.q.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4);
      const float4 G = ld4(B0 + i * PM + 4 * p), r = ld4(rr + (i / kSB) * DK + 4 * p);
      float4 kl, km, ql;
      for (int e = 0; e < 4; ++e) {
        const float lam = KB_EXP(comp(G, e) - comp(r, e)), mu = KB_EXP(comp(r, e) - comp(G, e));
        comp(kl, e) = comp(kv[u], e) * lam;
        comp(km, e) = comp(kv[u], e) * mu;
        comp(ql, e) = comp(qv[u], e) * lam;
      }
      st4(B1 + i * PM + 4 * p, kl);
      st4(B2 + i * PM + 4 * p, km);
      st4(B3 + i * PM + 4 * p, ql);
    }
  }
  for (int idx = tid; idx < 10 * DK; idx += NT) {
    const int p = idx / DK, d = idx - p * DK;
    const int I = p >= 6 ? 3 : p >= 3 ? 2 : p >= 1 ? 1 : 0;
    const int J = p - I * (I + 1) / 2;
    tau[idx] = KB_EXP(rr[I * DK + d] - rr[J * DK + d]);
  }
  KB_SYNC();
  // 3. Gram matrices A (strict) and A_Q (inclusive), one 4 x 4 tile per thread;
  //    T starts as zero
  {
    const int it = tid / 16, jt = tid % 16;
    float acc[4][4], accq[4][4];
    for (int r = 0; r < 4; ++r)
      for (int c = 0; c < 4; ++c) acc[r][c] = accq[r][c] = 0.f;
    if (jt <= it) {
      const int I = it / 4, J = jt / 4;
      const float* tp = tau + (I * (I + 1) / 2 + J) * DK;
      for (int d = 0; d < DK; d += 4) {
        const float4 t4 = ld4(tp + d);
        float4 kr[4];
        for (int c = 0; c < 4; ++c) {
          kr[c] = ld4(B2 + (4 * jt + c) * PM + d);
          kr[c].x *= t4.x;
          kr[c].y *= t4.y;
          kr[c].z *= t4.z;
          kr[c].w *= t4.w;
        }
        for (int r = 0; r < 4; ++r) {
          const float4 kl = ld4(B1 + (4 * it + r) * PM + d);
          const float4 ql = ld4(B3 + (4 * it + r) * PM + d);
          for (int c = 0; c < 4; ++c) {
            acc[r][c] += kl.x * kr[c].x + kl.y * kr[c].y + kl.z * kr[c].z + kl.w * kr[c].w;
            accq[r][c] += ql.x * kr[c].x + ql.y * kr[c].y + ql.z * kr[c].z + ql.w * kr[c].w;
          }
        }
      }
    }
    for (int r = 0; r < 4; ++r)
      for (int c = 0; c < 4; ++c) {
        const int i = 4 * it + r, j = 4 * jt + c;
        sA[i * PA + j] = j < i ? acc[r][c] : 0.f;
        sAQ[i * PA + j] = j <= i ? accq[r][c] : 0.f;
        sT[i * PA + j] = 0.f;
      }
  }
  KB_SYNC();
  // 4. T = (I + diag(beta) A)^-1
  invert_lower<NT>(sA, sT, sb, B0, PA, PM, tid);
  // 5. elementwise: B3 <- diag(beta) K+, B2 <- K_end, B0 <- scale Q+; records
  //    K_end, diag(beta) K+, e^{G_C} and A
  for (int idx = tid; idx < kC * DK; idx += NT) {
    const int i = idx / DK, d = idx - i * DK, I = i / kSB;
    const float r = rr[I * DK + d], gc = rr[4 * DK + d];
    const float er = KB_EXP(r), egr = KB_EXP(gc - r);
    const float kbv = sb[i] * B1[i * PM + d] * er;
    const float ke = B2[i * PM + d] * egr;
    const float qs = scale * B3[i * PM + d] * er;
    B3[i * PM + d] = kbv;
    B2[i * PM + d] = ke;
    B0[i * PM + d] = qs;
    rec[R::KE + i * DK + d] = ke;
    rec[R::KB + i * DK + d] = kbv;
  }
  for (int d = tid; d < DK; d += NT) rec[R::EGC + d] = KB_EXP(rr[4 * DK + d]);
  for (int idx = tid; idx < kC * kC; idx += NT) {
    const int i = idx / kC, j = idx - i * kC;
    rec[R::A + idx] = sA[i * PA + j];
  }
  KB_SYNC();
  // 6. W = T (diag(beta) K+), W_y = T^T K_end; dO into B1
  const int rg = tid / 16, cg = tid % 16;
  {
    float4 acc[4][DK / 64];
    zero_acc<DK>(acc);
    mm64_rows<DK>(acc, sT, PA, B3, PM, 0, 4 * rg + 4, rg, cg);
    store64<DK>(rec + R::W, DK, acc, rg, cg);
    zero_acc<DK>(acc);
    mm64_cols<DK>(acc, sT, PA, B2, PM, 4 * rg, kC, rg, cg);
    store64<DK>(rec + R::WY, DK, acc, rg, cg);
  }
  {
    float4 ov[NV];
    load_rows<DV, NT, T>(ov, ob, ba.dout.st, rows, tid);
    for (int u = 0; u < NV; ++u) {
      const int idx = tid + u * NT, i = idx / (DV / 4), p = idx - i * (DV / 4);
      st4(B1 + i * PM + 4 * p, ov[u]);
    }
  }
  KB_SYNC();
  // 7. Z_q = (scale Q+)^T dO; V_t = scale A_Q^T dO into B2; diag(beta) V into B3
  {
    // [DK][DV] result: rows {4 rg + 64 r4 + e}, columns {4 cg + 64 c4 + e}
    float4 acc[DK / 64][4][DV / 64];
    for (int r4 = 0; r4 < DK / 64; ++r4)
      for (int e = 0; e < 4; ++e)
        for (int c4 = 0; c4 < DV / 64; ++c4) acc[r4][e][c4] = zero4();
    for (int i = 0; i < kC; ++i) {
      float4 ov[DV / 64];
      for (int c4 = 0; c4 < DV / 64; ++c4) ov[c4] = ld4(B1 + i * PM + 4 * cg + 64 * c4);
      for (int r4 = 0; r4 < DK / 64; ++r4) {
        float4 qv = ld4(B0 + i * PM + 4 * rg + 64 * r4);
        for (int e = 0; e < 4; ++e)
          for (int c4 = 0; c4 < DV / 64; ++c4) fma4(acc[r4][e][c4], comp(qv, e), ov[c4]);
      }
    }
    for (int r4 = 0; r4 < DK / 64; ++r4)
      for (int e = 0; e < 4; ++e)
        for (int c4 = 0; c4 < DV / 64; ++c4)
          st4(rec + R::ZQ + (int64_t)(4 * rg + 64 * r4 + e) * DV + 4 * cg + 64 * c4, acc[r4][e][c4]);
  }
  {
    float4 acc[4][DV / 64];
    zero_acc<DV>(acc);
    mm64_cols<DV>(acc, sAQ, PA, B1, PM, 4 * rg, kC, rg, cg);
    for (int r = 0; r < 4; ++r)
      for (int c4 = 0; c4 < DV / 64; ++c4) {
        float4 x = acc[r][c4];
        x.x *= scale;
        x.y *= scale;
        x.z *= scale;
        x.w *= scale;
        st4(B2 + (4 * rg + r) * PM + 4 * cg + 64 * c4, x);
      }
  }
  {
    float4 vv[NV];
    load_rows<DV, NT, T>(vv, vb, a.v.st, rows, tid);
    for (int u = 0; u < NV; ++u) {
      const int idx = tid + u * NT, i = idx / (DV / 4), p = idx - i * (DV / 4);
      const float be = sb[i];
      float4 x = vv[u];
      x.x *= be;
      x.y *= be;
      x.z *= be;
      x.w *= be;
      st4(B3 + i * PM + 4 * p, x);
    }
  }
  KB_SYNC();
  // 8. V_y = T^T V_t, U_bar = T diag(beta) V
  {
    float4 acc[4][DV / 64];
    zero_acc<DV>(acc);
    mm64_cols<DV>(acc, sT, PA, B2, PM, 4 * rg, kC, rg, cg);
    store64<DV>(rec + R::VY, DV, acc, rg, cg);
    zero_acc<DV>(acc);
    mm64_rows<DV>(acc, sT, PA, B3, PM, 0, 4 * rg + 4, rg, cg);
    store64<DV>(rec + R::UB, DV, acc, rg, cg);
  }
}


// ---------------------------------------------------------------------------
// forward and reverse state passes: one CTA of 256 threads per (sequence, head,
// 32 value columns); the next chunk's record slice is copied in while the
// current one is used
constexpr int kPassThreads = 256;

template <int DK>
struct PassSmem {
  static constexpr int PK = DK + 4, PW = kW + 4;
  // one record buffer: two [64][DK] matrices, a [64][32] slice, a [DK][32] slice
  // (reverse pass only) and e^{G_C}
  static constexpr int M0 = 0, M1 = kC * PK, V0 = 2 * kC * PK, Z0 = V0 + kC * PW, E0 = Z0 + DK * PW;
  static constexpr int BUF = E0 + DK;
  static constexpr int ST = 2 * BUF;      // [DK][32] state (or state gradient) slice
  static constexpr int Y = ST + DK * PW;  // [64][32] U (forward) or dY (reverse)
  static constexpr int P = Y + kC * PW;   // [64][32] second half of the contraction over d_k
  static constexpr int FLOATS = P + kC * PW;
  static constexpr int BYTES = FLOATS * 4;
};

template <int DK, int DV>
KB_HD void pass_load(float* buf, const float* rec, int col0, bool reverse, int tid) {
  constexpr int NT = kPassThreads;
  using P = PassSmem<DK>;
  using R = Rec<DK, DV>;
  const float* m0 = rec + (reverse ? R::WY : R::W);
  const float* m1 = rec + (reverse ? R::KB : R::KE);
  const float* v0 = rec + (reverse ? R::VY : R::UB);
  for (int idx = tid; idx < kC * DK / 4; idx += NT) {
    const int i = idx / (DK / 4), p = idx - i * (DK / 4);
    cp16(buf + P::M0 + i * P::PK + 4 * p, m0 + i * DK + 4 * p);
    cp16(buf + P::M1 + i * P::PK + 4 * p, m1 + i * DK + 4 * p);
  }
  for (int idx = tid; idx < kC * kW / 4; idx += NT) {
    const int i = idx / (kW / 4), p = idx - i * (kW / 4);
    cp16(buf + P::V0 + i * P::PW + 4 * p, v0 + i * DV + col0 + 4 * p);
  }
  if (reverse)
    for (int idx = tid; idx < DK * kW / 4; idx += NT) {
      const int d = idx / (kW / 4), p = idx - d * (kW / 4);
      cp16(buf + P::Z0 + d * P::PW + 4 * p, rec + R::ZQ + d * DV + col0 + 4 * p);
    }
  for (int idx = tid; idx < DK / 4; idx += NT) cp16(buf + P::E0 + 4 * idx, rec + R::EGC + 4 * idx);
}

// reverse = false: S_c and U of every chunk.  reverse = true: X_c and dY of every
// chunk (chunks in reverse), dv = diag(beta) dY and the initial-state gradient.
template <int DK, int DV, typename T, bool reverse>
KB_HD void pass_body(const ChunkBwdArgs& ca, float* sm, int blk, int tid) {
  constexpr int NT = kPassThreads;
  using P = PassSmem<DK>;
  using R = Rec<DK, DV>;
  constexpr int PK = P::PK, PW = P::PW;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  constexpr int nsl = DV / kW;
  const int sl = blk % nsl, nh = blk / nsl;
  const int n = nh / a.H, h = nh - n * a.H;
  const int col0 = sl * kW;
  int64_t b, t0;
  int len;
  seq_span(a, n, b, t0, len);
  const int nc = num_chunks(ca, n), f0 = first_chunk(ca, n);
  float* sS = sm + P::ST;
  float* sY = sm + P::Y;
  float* sP = sm + P::P;
  // starting state: S_0 (forward) or the final-state gradient (reverse); zero if absent
  const float* init = reverse ? (ba.dsT ? ba.dsT + n * ba.dsT_sn + h * ba.dsT_sh : nullptr)
                              : (a.s0 ? a.s0 + n * a.s0_sn + h * a.s0_sh : nullptr);
  for (int idx = tid; idx < DK * kW; idx += NT) {
    const int d = idx / kW, v = idx - d * kW;
    sS[d * PW + v] = init ? init[(int64_t)d * DV + col0 + v] : 0.f;
  }
  auto recp = [&](int c) { return ca.rec + ((int64_t)(f0 + c) * a.H + h) * R::SIZE; };
  auto stp = [&](int c) { return ca.st + ((int64_t)(f0 + c) * a.H + h) * R::SSIZE; };
  if (nc > 0) pass_load<DK, DV>(sm, recp(reverse ? nc - 1 : 0), col0, reverse, tid);
  cp_commit();
  // first product: [64][32] tiles of 4 x 4 (rows 4 rg.., columns 4 cg..), each half
  // of the CTA over one half of d_k
  const int half = tid / 128, t = tid % 128, rg = t / 8, cg = t % 8;
  for (int k = 0; k < nc; ++k) {
    const int c = reverse ? nc - 1 - k : k;
    float* buf = sm + (k & 1) * P::BUF;
    cp_wait_all();
    KB_SYNC();
    if (k + 1 < nc) pass_load<DK, DV>(sm + ((k + 1) & 1) * P::BUF, recp(reverse ? c - 1 : c + 1), col0, reverse, tid);
    cp_commit();
    float* st = stp(c);
    // the state slice entering this step, to the chunk's state record
    for (int idx = tid; idx < DK * kW / 4; idx += NT) {
      const int d = idx / (kW / 4), p = idx - d * (kW / 4);
      st4(st + (reverse ? R::X : R::S) + (int64_t)d * DV + col0 + 4 * p, ld4(sS + d * PW + 4 * p));
    }
    // M0 S over this half of d_k: into sY (first half) or sP (second half)
    {
      float4 acc[4];
      for (int r = 0; r < 4; ++r) acc[r] = zero4();
      const int d0 = half * (DK / 2);
      for (int d = d0; d < d0 + DK / 2; d += 4) {
        float4 s4[4];
        for (int e = 0; e < 4; ++e) s4[e] = ld4(sS + (d + e) * PW + 4 * cg);
        for (int r = 0; r < 4; ++r) {
          const float4 m = ld4(buf + P::M0 + (4 * rg + r) * PK + d);
          for (int e = 0; e < 4; ++e) fma4(acc[r], comp(m, e), s4[e]);
        }
      }
      float* dst = half ? sP : sY;
      for (int r = 0; r < 4; ++r) st4(dst + (4 * rg + r) * PW + 4 * cg, acc[r]);
    }
    KB_SYNC();
    // Y = V0 -/+ M0 S  (forward: U = U_bar - W S; reverse: dY = V_y + W_y X)
    for (int idx = tid; idx < kC * kW / 4; idx += NT) {
      const int i = idx / (kW / 4), p = idx - i * (kW / 4);
      const float4 v0 = ld4(buf + P::V0 + i * PW + 4 * p), p0 = ld4(sY + i * PW + 4 * p),
                   p1 = ld4(sP + i * PW + 4 * p);
      const float sg = reverse ? 1.f : -1.f;
      float4 y;
      y.x = v0.x + sg * (p0.x + p1.x);
      y.y = v0.y + sg * (p0.y + p1.y);
      y.z = v0.z + sg * (p0.z + p1.z);
      y.w = v0.w + sg * (p0.w + p1.w);
      st4(sY + i * PW + 4 * p, y);
      st4(st + (reverse ? R::DY : R::U) + (int64_t)i * DV + col0 + 4 * p, y);
      if (reverse && i < len - c * kC) {  // dv = beta dY on valid rows
        const int64_t tok = t0 + (int64_t)c * kC + i;
        const float be = a.beta[b * a.beta_sb + tok * a.beta_st + (int64_t)h * a.beta_sh];
        float4 dv;
        dv.x = be * y.x;
        dv.y = be * y.y;
        dv.z = be * y.z;
        dv.w = be * y.w;
        st4(ba.dv.ptr + b * ba.dv.sb + tok * ba.dv.st + (int64_t)h * ba.dv.sh + col0 + 4 * p, dv);
      }
    }
    KB_SYNC();
    // state step on [DK][32] tiles of 4 x 4 (rows 4 dg.., columns 4 vg..):
    // S <- e^{G_C} S + K_end^T U, or X <- e^{G_C} X + Z_q - (diag(beta) K+)^T dY
    if (tid < 2 * DK) {
      const int dg = tid / 8, vg = tid % 8;
      float4 acc[4];
      for (int e = 0; e < 4; ++e) acc[e] = zero4();
      for (int i = 0; i < kC; ++i) {
        const float4 y = ld4(sY + i * PW + 4 * vg);
        const float4 m = ld4(buf + P::M1 + i * PK + 4 * dg);
        for (int e = 0; e < 4; ++e) fma4(acc[e], comp(m, e), y);
      }
      for (int e = 0; e < 4; ++e) {
        const int d = 4 * dg + e;
        const float eg = buf[P::E0 + d];
        float4 sv = ld4(sS + d * PW + 4 * vg);
        const float4 z = reverse ? ld4(buf + P::Z0 + d * PW + 4 * vg) : zero4();
        const float sg = reverse ? -1.f : 1.f;
        sv.x = eg * sv.x + z.x + sg * acc[e].x;
        sv.y = eg * sv.y + z.y + sg * acc[e].y;
        sv.z = eg * sv.z + z.z + sg * acc[e].z;
        sv.w = eg * sv.w + z.w + sg * acc[e].w;
        st4(sS + d * PW + 4 * vg, sv);
      }
    }
  }
  cp_wait_all();
  if (reverse && ba.ds0) {
    KB_SYNC();
    float* dst = ba.ds0 + n * ba.ds0_sn + h * ba.ds0_sh;
    for (int idx = tid; idx < DK * kW / 4; idx += NT) {
      const int d = idx / (kW / 4), p = idx - d * (kW / 4);
      st4(dst + (int64_t)d * DV + col0 + 4 * p, ld4(sS + d * PW + 4 * p));
    }
  }
}

// ---------------------------------------------------------------------------
// gradients of one chunk: one CTA of 256 threads per (chunk index, head).
//
// With R = V - K+ S, dY = T^T dU (from the reverse pass) and dR = diag(beta) dY:
//   dv    = dR (written by the reverse pass)
//   dbeta = rowsum(dY * (R - A U))                       (A strictly lower)
//   M1    = scale Tril(dO U^T),  M2 = -StrictTril(dR U^T)  (dA_Q and dA)
//   dq    = scale (dO S^T) e^G + sum_{j<=i} M1_ij k_j e^{G_i - G_j}
//   dk    = -(dR S^T) e^G + (U X^T) e^{G_C - G} + sum_{j<i} M2_ij k_j e^{G_i - G_j}
//           + sum_{i>=j} (M1_ij q_i + M2_ij k_i) e^{G_i - G_j}      (at row j)
//   dG    = (a - b - e) k + dq q with a, b, e the three kinds of dk terms above
//   dg    = reverse cumulative sum of dG + e^{G_C} rowsum(S X) + sum_t e_t k_t
template <int DK, int DV>
struct GradSmem {
  static constexpr int PK = DK + 4, PA = kC + 4, PB = 17;
  static constexpr int G = 0;                      // [64][PK] cumulative log-decay
  static constexpr int OP = G + kC * PK;           // [64][PK] K+, then k e^{r - G}, q e^{G - c}, dG
  static constexpr int A = OP + kC * PK;           // [64][PA]
  static constexpr int SL = A + kC * PA;           // slice buffers, later M1, M2, k e^{G - c}
  static constexpr int ST = SL, XT = ST + kW * PK;                  // [32][PK] S^T, X^T slices
  static constexpr int UT = XT + kW * PK, YT = UT + kW * PA;        // [32][PA] U^T, dY^T slices
  static constexpr int OT = YT + kW * PA, VT = OT + kW * PA;        // [32][PA] dO^T, V^T slices
  static constexpr int M1 = SL, M2 = M1 + kC * PA, OP2 = M2 + kC * PA;
  static constexpr int SLEND = VT + kW * PA;
  static_assert(OP2 + kC * PK == SLEND, "slice and after-slice layouts cover the same floats");
  static constexpr int RR = SLEND;                 // [5][DK]: r_0..r_3, G_C (= c_3); c_I = r_{I+1}
  static constexpr int BETA = RR + 5 * DK;         // [64]
  static constexpr int DBP = BETA + kC;            // [64][PB] dbeta partials
  static constexpr int EK = DBP + kC * PB;         // [16][DK] sum over 4 rows of e k
  static constexpr int GS = EK + 16 * DK;          // [DK] rowsum(S X)
  static constexpr int FLOATS = GS + DK;
  static constexpr int BYTES = FLOATS * 4;
};

// Shared-memory arrays of the second half of the gradient kernels (fp32; row pitches
// in floats).
struct TailSmem {
  float* G;     // [64][pg] cumulative log-decay G
  float* rr;    // [5][DK] r_0 .. r_3 (log-decay before each sub-block), G_C
  float* beta;  // [64]
  float* M1;    // [64][pm] scale Tril(dO U^T)
  float* M2;    // [64][pm] -StrictTril(diag(beta) dY U^T)
  float* op;    // [64][po] operand buffer, then dG
  float* op2;   // [64][po] operand buffer
  float* ek;    // [16][DK] sums over 4 rows of e k
  float* dbp;   // [64][pb] dbeta partials, nb per row
  float* gs;    // [DK] rowsum(S X)
  int pg, pm, po, pb, nb;
};

// Second half of the gradients of one chunk, from Pq = dO S^T, Pk = dY S^T and
// Pe = U X^T (a thread's rows 4 rg .., columns 4 cg + 64 c4 ..) and M1, M2, gs and
// the dbeta partials in shared memory: the direct terms, the row and column forms
// inside the chunk, dq, dk, dg and dbeta.  With kp_dbeta the term
// -rowsum(K+ * (dY S^T)) of dbeta is formed here, as partial cg of each row.
template <int DK, int DV, typename T, bool kp_dbeta>
KB_HD void grad_tail(const ChunkBwdArgs& ca, const ChunkLoc& L, int h, const TailSmem& s,
                     float4 (&Pq)[4][DK / 64], float4 (&Pk)[4][DK / 64], float4 (&Pe)[4][DK / 64], int tid) {
  constexpr int NT = 256;
  constexpr int C4 = DK / 64;
  constexpr int NK = kC * DK / 4 / NT;  // 4-vectors of a [64][DK] tile per thread
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  const T* qb = static_cast<const T*>(a.q.ptr) + L.b * a.q.sb + L.t * a.q.st + (int64_t)h * a.q.sh;
  const T* kb = static_cast<const T*>(a.k.ptr) + L.b * a.k.sb + L.t * a.k.st + (int64_t)h * a.k.sh;
  const int rows = L.rows;
  const float scale = a.scale;
  const int rg = tid / 16, cg = tid % 16;
  const int PG = s.pg, PA = s.pm, PO = s.po;
  float* sG = s.G;
  float* rr = s.rr;
  float* sb = s.beta;
  float* sM1 = s.M1;
  float* sM2 = s.M2;
  float* sOp = s.op;
  float* sOp2 = s.op2;
  float* ek = s.ek;
  auto own = [&](float4 (&x)[4][C4], const T* base, int64_t st) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c4 = 0; c4 < C4; ++c4)
        x[r][c4] = 4 * rg + r < rows ? ld4t<T>(base + (int64_t)(4 * rg + r) * st + 4 * cg + 64 * c4) : zero4();
  };
  // direct terms; after this block Pq = dq, Pk = dk, Pe = (a - e) (the dG coefficient of k)
  float4 kown[4][C4];
  own(kown, kb, a.k.st);
  float dbk[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c4 = 0; c4 < C4; ++c4)
    for (int e = 0; e < 4; ++e) {
      const int d = 4 * cg + 64 * c4 + e;
      float eks = 0.f;
      for (int r = 0; r < 4; ++r) {
        const int i = 4 * rg + r;
        const float G = sG[i * PG + d];
        const float E = KB_EXP(G), Ee = KB_EXP(rr[4 * DK + d] - G);
        if (kp_dbeta) dbk[r] += comp(kown[r][c4], e) * E * comp(Pk[r][c4], e);
        const float dq = scale * comp(Pq[r][c4], e) * E;
        const float av = -sb[i] * comp(Pk[r][c4], e) * E;
        const float ev = comp(Pe[r][c4], e) * Ee;
        comp(Pq[r][c4], e) = dq;
        comp(Pk[r][c4], e) = av + ev;
        comp(Pe[r][c4], e) = av - ev;
        eks += ev * comp(kown[r][c4], e);
      }
      ek[rg * DK + d] = eks;
    }
  if (kp_dbeta)
    for (int r = 0; r < 4; ++r) s.dbp[(4 * rg + r) * s.pb + cg] = -dbk[r];
  {
    float4 kv[NK];
    load_rows<DK, NT, T>(kv, kb, a.k.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4), I = i / kSB;
      const float4 G = ld4(sG + i * PG + 4 * p);
      const float4 r0 = ld4(rr + I * DK + 4 * p), r1 = ld4(rr + (I + 1) * DK + 4 * p);
      float4 x, y;
      for (int e = 0; e < 4; ++e) {
        comp(x, e) = comp(kv[u], e) * KB_EXP(comp(r0, e) - comp(G, e));
        comp(y, e) = comp(kv[u], e) * KB_EXP(comp(G, e) - comp(r1, e));
      }
      st4(sOp + i * PO + 4 * p, x);
      st4(sOp2 + i * PO + 4 * p, y);
    }
  }
  KB_SYNC();
  // row form: sum_{j in J} M_ij (k_j e^{r_J - G_j}), times e^{G_i - r_J}
  const int Ib = rg / 4;  // the sub-block of this thread's rows
  for (int pass = 0; pass < 2; ++pass) {
    const float* M = pass ? sM2 : sM1;
    for (int J = 0; J <= Ib; ++J) {
      float4 t[4][C4];
      zero_acc<DK>(t);
      mm64_rows<DK>(t, M, PA, sOp, PO, kSB * J, kSB * J + kSB, rg, cg);
      for (int r = 0; r < 4; ++r)
        for (int c4 = 0; c4 < C4; ++c4)
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * rg + r, d = 4 * cg + 64 * c4 + e;
            const float x = KB_EXP(sG[i * PG + d] - rr[J * DK + d]) * comp(t[r][c4], e);
            if (pass == 0) {
              comp(Pq[r][c4], e) += x;
            } else {
              comp(Pk[r][c4], e) += x;
              comp(Pe[r][c4], e) += x;
            }
          }
    }
  }
  KB_SYNC();
  {
    float4 qv[NK];
    load_rows<DK, NT, T>(qv, qb, a.q.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4);
      const float4 G = ld4(sG + i * PG + 4 * p), r1 = ld4(rr + (i / kSB + 1) * DK + 4 * p);
      float4 x;
      for (int e = 0; e < 4; ++e) comp(x, e) = comp(qv[u], e) * KB_EXP(comp(G, e) - comp(r1, e));
      st4(sOp + i * PO + 4 * p, x);
    }
  }
  KB_SYNC();
  // column form at rows j: sum_{i in I} (M1_ij q_i + M2_ij k_i) e^{G_i - c_I}, times e^{c_I - G_j}
  for (int I = Ib; I < 4; ++I) {
    float4 t[4][C4];
    zero_acc<DK>(t);
    mm64_cols<DK>(t, sM1, PA, sOp, PO, kSB * I, kSB * I + kSB, rg, cg);
    mm64_cols<DK>(t, sM2, PA, sOp2, PO, kSB * I, kSB * I + kSB, rg, cg);
    for (int r = 0; r < 4; ++r)
      for (int c4 = 0; c4 < C4; ++c4)
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * rg + r, d = 4 * cg + 64 * c4 + e;
          const float x = KB_EXP(rr[(I + 1) * DK + d] - sG[j * PG + d]) * comp(t[r][c4], e);
          comp(Pk[r][c4], e) += x;
          comp(Pe[r][c4], e) -= x;
        }
  }
  KB_SYNC();
  // dq, dk out; dG = (a - b - e) k + dq q into sOp
  float4 qown[4][C4];
  own(kown, kb, a.k.st);
  own(qown, qb, a.q.st);
  for (int r = 0; r < 4; ++r) {
    const int i = 4 * rg + r;
    for (int c4 = 0; c4 < C4; ++c4) {
      float4 dg4;
      for (int e = 0; e < 4; ++e)
        comp(dg4, e) = comp(Pe[r][c4], e) * comp(kown[r][c4], e) + comp(Pq[r][c4], e) * comp(qown[r][c4], e);
      st4(sOp + i * PO + 4 * cg + 64 * c4, dg4);
      if (i < rows) {
        const int64_t t = L.t + i;
        st4(ba.dq.ptr + L.b * ba.dq.sb + t * ba.dq.st + (int64_t)h * ba.dq.sh + 4 * cg + 64 * c4, Pq[r][c4]);
        st4(ba.dk.ptr + L.b * ba.dk.sb + t * ba.dk.st + (int64_t)h * ba.dk.sh + 4 * cg + 64 * c4, Pk[r][c4]);
      }
    }
  }
  KB_SYNC();
  // dg: reverse cumulative sum down the chunk plus the G_C terms; dbeta
  for (int d = tid; d < DK; d += NT) {
    float run = KB_EXP(rr[4 * DK + d]) * s.gs[d];
    for (int q = 0; q < 16; ++q) run += ek[q * DK + d];
    for (int i = rows - 1; i >= 0; --i) {
      run += sOp[i * PO + d];
      ba.dg.ptr[L.b * ba.dg.sb + (L.t + i) * ba.dg.st + (int64_t)h * ba.dg.sh + d] = run;
    }
  }
  for (int i = tid - (NT - kC); i >= 0 && i < rows; i += NT) {
    float acc = 0.f;
    for (int q = 0; q < s.nb; ++q) acc += s.dbp[i * s.pb + q];
    ba.dbeta[L.b * ba.db_sb + (L.t + i) * ba.db_st + (int64_t)h * ba.db_sh] = acc;
  }
}

template <int DK, int DV, typename T>
KB_HD void grad_body(const ChunkBwdArgs& ca, float* sm, int f, int h, int tid) {
  constexpr int NT = 256;
  constexpr int C4 = DK / 64;
  using SM = GradSmem<DK, DV>;
  using R = Rec<DK, DV>;
  constexpr int PK = SM::PK, PA = SM::PA;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  ChunkLoc L;
  if (!locate(ca, f, L)) return;  // uniform across the CTA
  const float* rec = ca.rec + ((int64_t)f * a.H + h) * R::SIZE;
  const float* stt = ca.st + ((int64_t)f * a.H + h) * R::SSIZE;
  const T* kb = static_cast<const T*>(a.k.ptr) + L.b * a.k.sb + L.t * a.k.st + (int64_t)h * a.k.sh;
  const T* vb = static_cast<const T*>(a.v.ptr) + L.b * a.v.sb + L.t * a.v.st + (int64_t)h * a.v.sh;
  const T* ob = static_cast<const T*>(ba.dout.ptr) + L.b * ba.dout.sb + L.t * ba.dout.st + (int64_t)h * ba.dout.sh;
  const float* gb = static_cast<const float*>(a.g.ptr) + L.b * a.g.sb + L.t * a.g.st + (int64_t)h * a.g.sh;
  const float* bb = a.beta + L.b * a.beta_sb + L.t * a.beta_st + (int64_t)h * a.beta_sh;
  float* sG = sm + SM::G;
  float* sOp = sm + SM::OP;
  float* sA = sm + SM::A;
  float* rr = sm + SM::RR;
  float* sb = sm + SM::BETA;
  const int rows = L.rows;
  const float scale = a.scale;
  constexpr int NK = kC * DK / 4 / NT;  // 4-vectors of a [64][DK] tile per thread
  const int rg = tid / 16, cg = tid % 16;

  // 1. log-decays, beta, A; cumulative sums and the sub-block references
  {
    float4 gv[NK];
    load_rows<DK, NT, float>(gv, gb, a.g.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4);
      st4(sG + i * PK + 4 * p, gv[u]);
    }
  }
  for (int i = tid; i < kC; i += NT) sb[i] = i < rows ? bb[(int64_t)i * a.beta_st] : 0.f;
  for (int idx = tid; idx < kC * kC; idx += NT) {
    const int i = idx / kC, j = idx - i * kC;
    sA[i * PA + j] = rec[R::A + idx];
  }
  KB_SYNC();
  for (int d = tid; d < DK; d += NT) {
    float run = 0.f;
    rr[d] = 0.f;
    for (int i = 0; i < kC; ++i) {
      run += sG[i * PK + d];
      sG[i * PK + d] = run;
      if ((i & (kSB - 1)) == kSB - 1) rr[((i + 1) / kSB) * DK + d] = run;
    }
  }
  KB_SYNC();
  // 2. K+ = k e^G
  {
    float4 kv[NK];
    load_rows<DK, NT, T>(kv, kb, a.k.st, rows, tid);
    for (int u = 0; u < NK; ++u) {
      const int idx = tid + u * NT, i = idx / (DK / 4), p = idx - i * (DK / 4);
      const float4 G = ld4(sG + i * PK + 4 * p);
      float4 x;
      for (int e = 0; e < 4; ++e) comp(x, e) = comp(kv[u], e) * KB_EXP(comp(G, e));
      st4(sOp + i * PK + 4 * p, x);
    }
  }

  float4 Pq[4][C4], Pk[4][C4], Pe[4][C4];  // dO S^T, dY S^T, U X^T
  float4 QA[4], YA[4];                     // dO U^T, dY U^T at columns 4 cg ..
  float dbp[4] = {0.f, 0.f, 0.f, 0.f};
  float gsum = 0.f;
  zero_acc<DK>(Pq);
  zero_acc<DK>(Pk);
  zero_acc<DK>(Pe);
  for (int r = 0; r < 4; ++r) QA[r] = YA[r] = zero4();
  float* sST = sm + SM::ST;
  float* sXT = sm + SM::XT;
  float* sUT = sm + SM::UT;
  float* sYT = sm + SM::YT;
  float* sOT = sm + SM::OT;
  float* sVT = sm + SM::VT;
  for (int s = 0; s < DV / kW; ++s) {
    const int col0 = s * kW;
    // 3. this slice's columns, transposed: S, X [DK][32] -> [32][DK]; U, dY, dO, V [64][32] -> [32][64]
    {
      constexpr int NS = DK * kW / 4 / NT, NR = kC * kW / 4 / NT;
      float4 sv[NS], xv[NS], uv[NR], yv[NR], ov[NR], vv[NR];
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        const int idx = tid + u * NT, d = idx / (kW / 4), p = idx - d * (kW / 4);
        sv[u] = ld4(stt + R::S + (int64_t)d * DV + col0 + 4 * p);
        xv[u] = ld4(stt + R::X + (int64_t)d * DV + col0 + 4 * p);
      }
#pragma unroll
      for (int u = 0; u < NR; ++u) {
        const int idx = tid + u * NT, i = idx / (kW / 4), p = idx - i * (kW / 4);
        uv[u] = ld4(stt + R::U + (int64_t)i * DV + col0 + 4 * p);
        yv[u] = ld4(stt + R::DY + (int64_t)i * DV + col0 + 4 * p);
        ov[u] = i < rows ? ld4t<T>(ob + (int64_t)i * ba.dout.st + col0 + 4 * p) : zero4();
        vv[u] = i < rows ? ld4t<T>(vb + (int64_t)i * a.v.st + col0 + 4 * p) : zero4();
      }
      for (int u = 0; u < NS; ++u) {
        const int idx = tid + u * NT, d = idx / (kW / 4), p = idx - d * (kW / 4);
        for (int e = 0; e < 4; ++e) {
          sST[(4 * p + e) * PK + d] = comp(sv[u], e);
          sXT[(4 * p + e) * PK + d] = comp(xv[u], e);
        }
      }
      for (int u = 0; u < NR; ++u) {
        const int idx = tid + u * NT, i = idx / (kW / 4), p = idx - i * (kW / 4);
        for (int e = 0; e < 4; ++e) {
          sUT[(4 * p + e) * PA + i] = comp(uv[u], e);
          sYT[(4 * p + e) * PA + i] = comp(yv[u], e);
          sOT[(4 * p + e) * PA + i] = comp(ov[u], e);
          sVT[(4 * p + e) * PA + i] = comp(vv[u], e);
        }
      }
    }
    KB_SYNC();
    // 4. dbeta partials: dY (V - K+ S - A U) at rows 4 rg.., columns cg and cg + 16
    {
      float z[4][2];
      for (int r = 0; r < 4; ++r)
        for (int c = 0; c < 2; ++c) z[r][c] = sVT[(cg + 16 * c) * PA + 4 * rg + r];
      for (int d = 0; d < DK; d += 4) {
        const float4 s0 = ld4(sST + cg * PK + d), s1 = ld4(sST + (cg + 16) * PK + d);
        for (int r = 0; r < 4; ++r) {
          const float4 kp = ld4(sOp + (4 * rg + r) * PK + d);
          z[r][0] -= kp.x * s0.x + kp.y * s0.y + kp.z * s0.z + kp.w * s0.w;
          z[r][1] -= kp.x * s1.x + kp.y * s1.y + kp.z * s1.z + kp.w * s1.w;
        }
      }
      for (int j = 0; j < 4 * rg + 4; j += 4) {
        const float4 u0 = ld4(sUT + cg * PA + j), u1 = ld4(sUT + (cg + 16) * PA + j);
        for (int r = 0; r < 4; ++r) {
          const float4 av = ld4(sA + (4 * rg + r) * PA + j);
          z[r][0] -= av.x * u0.x + av.y * u0.y + av.z * u0.z + av.w * u0.w;
          z[r][1] -= av.x * u1.x + av.y * u1.y + av.z * u1.z + av.w * u1.w;
        }
      }
      for (int r = 0; r < 4; ++r)
        dbp[r] += sYT[cg * PA + 4 * rg + r] * z[r][0] + sYT[(cg + 16) * PA + 4 * rg + r] * z[r][1];
    }
    // 5. contractions over this slice's value columns
    for (int v = 0; v < kW; ++v) {
      const float4 o4 = ld4(sOT + v * PA + 4 * rg), y4 = ld4(sYT + v * PA + 4 * rg);
      const float4 ui4 = ld4(sUT + v * PA + 4 * rg), uj4 = ld4(sUT + v * PA + 4 * cg);
      float4 s4[C4], x4[C4];
      for (int c4 = 0; c4 < C4; ++c4) {
        s4[c4] = ld4(sST + v * PK + 4 * cg + 64 * c4);
        x4[c4] = ld4(sXT + v * PK + 4 * cg + 64 * c4);
      }
      float ov[4] = {o4.x, o4.y, o4.z, o4.w}, yv[4] = {y4.x, y4.y, y4.z, y4.w};
      float uv[4] = {ui4.x, ui4.y, ui4.z, ui4.w};
      for (int r = 0; r < 4; ++r) {
        for (int c4 = 0; c4 < C4; ++c4) {
          fma4(Pq[r][c4], ov[r], s4[c4]);
          fma4(Pk[r][c4], yv[r], s4[c4]);
          fma4(Pe[r][c4], uv[r], x4[c4]);
        }
        fma4(QA[r], ov[r], uj4);
        fma4(YA[r], yv[r], uj4);
      }
    }
    for (int d = tid; d < DK; d += NT)
      for (int v = 0; v < kW; ++v) gsum += sST[v * PK + d] * sXT[v * PK + d];
    KB_SYNC();
  }
  // 6. M1 = scale Tril(dO U^T), M2 = -StrictTril(diag(beta) dY U^T), the dbeta
  //    partials and rowsum(S X); then the second half shared with the tensor-core kernel
  float* sM1 = sm + SM::M1;
  float* sM2 = sm + SM::M2;
  for (int r = 0; r < 4; ++r) {
    const int i = 4 * rg + r;
    sm[SM::DBP + i * SM::PB + cg] = dbp[r];
    for (int c = 0; c < 4; ++c) {
      const int j = 4 * cg + c;
      sM1[i * PA + j] = j <= i ? scale * comp(QA[r], c) : 0.f;
      sM2[i * PA + j] = j < i ? -sb[i] * comp(YA[r], c) : 0.f;
    }
  }
  for (int d = tid; d < DK; d += NT) sm[SM::GS + d] = gsum;
  TailSmem ts;
  ts.G = sG;
  ts.rr = rr;
  ts.beta = sb;
  ts.M1 = sM1;
  ts.M2 = sM2;
  ts.op = sOp;
  ts.op2 = sm + SM::OP2;
  ts.ek = sm + SM::EK;
  ts.dbp = sm + SM::DBP;
  ts.gs = sm + SM::GS;
  ts.pg = PK;
  ts.pm = PA;
  ts.po = PK;
  ts.pb = SM::PB;
  ts.nb = 16;
  grad_tail<DK, DV, T, false>(ca, L, h, ts, Pq, Pk, Pe, tid);
}

}  // namespace bwdc

// The prep, state-pass and gradient kernels with their products on the tensor cores
// (kda_backward_tc.cu): d_k = d_v = 128 with bf16 inputs.
bool chunk_grad_tc_supported(const PrefillArgs& a);
cudaError_t launch_chunk_prep_tc(const bwdc::ChunkBwdArgs& ca, cudaStream_t s);
cudaError_t launch_chunk_pass_tc(const bwdc::ChunkBwdArgs& ca, bool reverse, cudaStream_t s);
cudaError_t launch_chunk_grad_tc(const bwdc::ChunkBwdArgs& ca, cudaStream_t s);

}  // namespace kda
