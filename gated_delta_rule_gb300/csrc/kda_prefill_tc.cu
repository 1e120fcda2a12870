// Chunked KDA prefill on the sm_100-family tensor cores (tcgen05 + TMEM).
//
// One CTA of 128 threads runs one (sequence, head) from its first chunk to its
// last; the fp32 state S (d_k x d_v) lives in TMEM for the whole sequence.
// Per chunk of C = 64 tokens (the chunked form of "尝试对Kimi KDA的数学推导&
// 算子实现分析" (hjcheng0602.cn/blog/kdd), written with U = (I + L)^-1 B_beta (V - K+ S)):
//
//   G_t   = sum_{r <= t} g_r inside the chunk                          (eq. 9)
//   L     = StrictTril(B_beta K+ K-^T)                                  (eq. 51)
//   A_Q   = Tril(Q+ K-^T)   (inclusive; the read-out sums j <= t)       (eq. 57)
//   T     = (I + L)^-1                                                  (eq. 27)
//   W     = T B_beta K+ ,  U0 = T B_beta V      (S-independent)         (eq. 52)
//   U     = U0 - W S                                                    (eq. 52)
//   O     = scale (Q+ S + A_Q U)                                        (eq. 63)
//   S'    = Diag(e^{G_C}) S + (K e^{G_C - G})^T U                       (eqs. 64-66)
//
// Exponents are only ever formed as differences that stay inside a 16-token
// sub-block or decay toward the later token, so nothing overflows for
// g in [-5, 0] (the lower-bounded decay of "Kimi K3 技术报告解读"
// (marsggbo.github.io) §3.5: a 16-token cumulative log-decay stays in (-80, 0]):
//   * Gram blocks use, for output rows in sub-block I, the reference G at the
//     start of sub-block I: rows K_i e^{G_i - G_{16I-1}} (<= 1) and columns
//     K_j e^{G_{16I-1} - G_j} (<= 1 for earlier sub-blocks, < e^80 inside I).
//     The column operand therefore exists in 4 versions, one per I, and the
//     Gram is computed transposed (M = key rows j, N = query/key rows i).
//   * K+ = K e^{G}, Q+ = Q e^{G}, K e^{G_C - G} are all <= 1.
//
// Tensor-core products (bf16 operands, fp32 accumulators in TMEM):
//   Gram^T (4 x [128 x 32 x d_k]), W / U0 (T_beta times [K+ | V]),
//   [U0 - W S] (the serial product with the bf16 copy of S),
//   S += K_end^T U, O = [Q+ | A_Q] [S ; U].
// The triangular inverse T is computed in fp32 on the CUDA cores (16 x 16
// diagonal blocks by forward substitution, then block rows).
//
// Several M = 128 products only use 64 meaningful A rows: their descriptor
// window extends over a neighbouring tile, and the corresponding accumulator
// rows are never read (or are overwritten before they are read).
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }

template <int DK, int DV>
struct Smem {
  // G region: Gram operands (Y versions, X); after the Gram: solve workspace + T_beta
  static constexpr int kYver = 64 * DK * 2;  // one version: 64 rows x DK, bf16
  static constexpr int Y = 0;
  static constexpr int X = Y + 4 * kYver;  // 128 rows x DK
  static constexpr int kGram = X + 128 * DK * 2;
  static constexpr int kLd = 65;  // fp32 row stride of L and T
  static constexpr int kRd = 49;  // fp32 row stride of the block-row workspace
  static constexpr int SL = 0;
  static constexpr int ST = SL + 64 * kLd * 4;
  static constexpr int SR = ST + 64 * kLd * 4;
  static constexpr int T2 = align1k(SR + 16 * kRd * 4);  // T_beta, 64 x 64 bf16 (+ 8K window)
  static constexpr int kSolve = T2 + 2 * 64 * 64 * 2;
  static constexpr int kG = kGram > kSolve ? kGram : kSolve;
  // persistent tiles
  static constexpr int KP = align1k(kG);                         // K+ (MN-major), later U (MN-major)
  static constexpr int kKP = 64 * (DK > DV ? DK : DV) * 2;
  static constexpr int VT = KP + kKP;                            // V chunk (MN-major)
  static constexpr int AW = VT + 64 * DV * 2;                    // -W (K-major)
  static constexpr int OQ = AW + 64 * DK * 2;                    // [Q+ | A_Q] (K-major)
  static constexpr int KE = OQ + 64 * (DK + 64) * 2;             // K e^{G_C - G} (MN-major)
  static constexpr int SB = KE + 64 * DK * 2;                    // bf16 S (MN-major, DK rows)
  static constexpr int MISC = SB + DK * DV * 2;
  static constexpr int BETA = MISC;                              // 64 fp32
  static constexpr int PDEC = BETA + 64 * 4;                     // DK fp32: e^{G_C}
  static constexpr int BND = PDEC + DK * 4;                      // 5 x DK fp32 (log2 units)
  static constexpr int CARRY = BND + 5 * DK * 4;                 // parts x DK fp32
  static constexpr int kParts = kThreads / (DK / 2);
  static constexpr int MBAR = CARRY + kParts * DK * 4;
  static constexpr int TSLOT = MBAR + 8;
  static constexpr int FLAG = TSLOT + 4;
  static constexpr int kTotal = FLAG + 4;
  static constexpr int kAlloc = kTotal + 1024;  // slack to align the base to 1024 bytes
  static_assert(kAlloc <= 232448, "shared memory budget");
  static constexpr uint32_t kTmemCols = (128 + 2 * DV) <= 256 ? 256 : 512;
};

struct Ctx {
  uint32_t mbar;
  uint32_t phase;
  volatile int* flag;
  int* err;
};

// Wait for the last MMA commit; on a timeout record it and raise the abort flag.
__device__ __forceinline__ void wait_mma(Ctx& c) {
  if (!mbar_wait(c.mbar, c.phase)) {
    atomicOr(c.err, kErrTimeout);
    *c.flag = 1;
  }
  c.phase ^= 1u;
  fence_after_sync();
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) kda_chunk_prefill_kernel(PrefillArgs a) {
  using L = Smem<DK, DV>;
  constexpr int NP = DK / 2;          // channel pairs
  constexpr int TPT = 64 / L::kParts; // tokens per thread in the build
  constexpr int NBT = TPT / 16;       // sub-blocks per thread in the build

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* sL = reinterpret_cast<float*>(smem + L::SL);
  float* sT = reinterpret_cast<float*>(smem + L::ST);
  float* sR = reinterpret_cast<float*>(smem + L::SR);
  float* sBeta = reinterpret_cast<float*>(smem + L::BETA);
  float* sP = reinterpret_cast<float*>(smem + L::PDEC);
  float* sBnd = reinterpret_cast<float*>(smem + L::BND);
  float* sCarry = reinterpret_cast<float*>(smem + L::CARRY);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + L::FLAG);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const int n = blockIdx.x / a.H;
  const int h = blockIdx.x - n * a.H;

  int64_t brow = n, tok0 = 0, len = a.T;
  if (a.cu_seqlens) {
    brow = 0;
    const int c0 = min(max(__ldg(a.cu_seqlens + n), 0), a.T);
    const int c1 = min(max(__ldg(a.cu_seqlens + n + 1), c0), a.T);
    tok0 = c0;
    len = c1 - c0;
  }
  const int nchunks = (int)((len + kC - 1) / kC);

  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q.ptr) + brow * a.q.sb + tok0 * a.q.st + h * a.q.sh;
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k.ptr) + brow * a.k.sb + tok0 * a.k.st + h * a.k.sh;
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v.ptr) + brow * a.v.sb + tok0 * a.v.st + h * a.v.sh;
  const float* gg = static_cast<const float*>(a.g.ptr) + brow * a.g.sb + tok0 * a.g.st + h * a.g.sh;
  const float* bg = a.beta + brow * a.beta_sb + tok0 * a.beta_st + h * a.beta_sh;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + brow * a.out_sb + tok0 * a.out_st + h * a.out_sh;

  // ---- setup: barrier, TMEM, initial state ----
  if (tid == 0) {
    mbar_init(sbase + L::MBAR, 1);
    fence_mbar_init();
    *sFlag = 0;
  }
  if (warp == 0) tmem_alloc(sbase + L::TSLOT, L::kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);
  const uint32_t tG = tmem;             // Gram^T (128 cols), then W (DK cols)
  const uint32_t tX = tmem + 128;       // U0 / U / O   (DV cols)
  const uint32_t tS = tmem + 128 + DV;  // fp32 state   (DV cols)
  Ctx ctx{sbase + L::MBAR, 0u, sFlag, a.err};

  if (tid < DK) {  // lane c holds state row c
    const float* s0 = a.s0 ? a.s0 + n * a.s0_sn + h * a.s0_sh + (int64_t)tid * DV : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + c0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[i] = x.x;
        v[i + 1] = x.y;
        v[i + 2] = x.z;
        v[i + 3] = x.w;
      }
      tmem_st32(tS + lane_base + c0, v);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4(sbase + L::SB + sw128(tid, c0 + 8 * u, DK), pack_bf16(v[8 * u], v[8 * u + 1]),
                     pack_bf16(v[8 * u + 2], v[8 * u + 3]), pack_bf16(v[8 * u + 4], v[8 * u + 5]),
                     pack_bf16(v[8 * u + 6], v[8 * u + 7]));
    }
  }

  // ---- per-thread build registers: channel pair p, tokens [part*TPT, +TPT) ----
  const int p = tid % NP;
  const int part = tid / NP;
  uint32_t rk[TPT], rq[TPT];
  float2 rg[TPT];
  float rbeta = 0.f;

  auto prefetch = [&](int ci) {
    const int64_t base = (int64_t)ci * kC;
    const int lc = (int)(len - base < kC ? len - base : kC);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = part * TPT + i;
      if (t < lc) {
        const int64_t row = base + t;
        rk[i] = __ldg(reinterpret_cast<const uint32_t*>(kg + row * a.k.st) + p);
        rq[i] = __ldg(reinterpret_cast<const uint32_t*>(qg + row * a.q.st) + p);
        rg[i] = __ldg(reinterpret_cast<const float2*>(gg + row * a.g.st) + p);
      } else {
        rk[i] = 0u;
        rq[i] = 0u;
        rg[i] = make_float2(0.f, 0.f);
      }
    }
    rbeta = (tid < lc) ? __ldg(bg + (base + tid) * a.beta_st) : 0.f;
  };
  auto prefetch_v = [&](int ci) {
    const int64_t base = (int64_t)ci * kC;
    const int lc = (int)(len - base < kC ? len - base : kC);
    constexpr int kVec = DV / 8;  // 16-byte vectors per row
#pragma unroll
    for (int it = 0; it < (64 * kVec) / kThreads; ++it) {
      const int idx = it * kThreads + tid;
      const int t = idx / kVec, cv = idx % kVec;
      const bool ok = t < lc;
      const __nv_bfloat16* src = ok ? vg + (base + t) * a.v.st + 8 * cv : vg;
      cp_async16(sbase + L::VT + sw128(t, 8 * cv, 64), src, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  if (nchunks > 0) {
    prefetch(0);
    prefetch_v(0);
  }

  for (int ci = 0; ci < nchunks; ++ci) {
    const int lc = (int)(len - (int64_t)ci * kC < kC ? len - (int64_t)ci * kC : kC);

    // ================= build: in-chunk scan and operand tiles =================
    float2 G[TPT];
    {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        acc.x += rg[i].x * kLog2e;
        acc.y += rg[i].y * kLog2e;
        G[i] = acc;
      }
      sCarry[part * DK + 2 * p] = acc.x;
      sCarry[part * DK + 2 * p + 1] = acc.y;
      if (tid < 64) sBeta[tid] = rbeta;
    }
    __syncthreads();
    {
      float2 off = make_float2(0.f, 0.f);
      for (int q = 0; q < part; ++q) {
        off.x += sCarry[q * DK + 2 * p];
        off.y += sCarry[q * DK + 2 * p + 1];
      }
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        G[i].x += off.x;
        G[i].y += off.y;
      }
      if (part == 0) {
        sBnd[2 * p] = 0.f;
        sBnd[2 * p + 1] = 0.f;
      }
#pragma unroll
      for (int b = 0; b < NBT; ++b) {
        const int kb = part * NBT + b + 1;  // boundary after this thread's sub-block b
        sBnd[kb * DK + 2 * p] = G[16 * b + 15].x;
        sBnd[kb * DK + 2 * p + 1] = G[16 * b + 15].y;
        if (kb == 4) {
          sP[2 * p] = exp2f(G[16 * b + 15].x);
          sP[2 * p + 1] = exp2f(G[16 * b + 15].y);
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < NBT; ++b) {
      const int I = part * NBT + b;
      float bl[2], fbl[2], hI[2], fke[2], fy[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 2 * p + e;
        bl[e] = sBnd[I * DK + c];
        const float en = sBnd[(I + 1) * DK + c];
        fbl[e] = exp2f(bl[e]);
        hI[e] = exp2f(en - bl[e]);
        fke[e] = exp2f(sBnd[4 * DK + c] - en);
#pragma unroll
        for (int J = 0; J < 4; ++J) fy[e][J] = (J > I) ? exp2f(sBnd[J * DK + c] - en) : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int i = 16 * b + r;
        const int t = part * TPT + i;
        const float k0 = bf_lo(rk[i]), k1 = bf_hi(rk[i]);
        const float q0 = bf_lo(rq[i]), q1 = bf_hi(rq[i]);
        const float a0 = exp2f(G[i].x - bl[0]), a1 = exp2f(G[i].y - bl[1]);
        const float ia0 = exp2f(bl[0] - G[i].x), ia1 = exp2f(bl[1] - G[i].y);
        const float e0 = hI[0] * ia0, e1 = hI[1] * ia1;
        const uint32_t col = 2 * p;
        st_shared_u32(sbase + L::KP + sw128(t, col, 64), pack_bf16(k0 * a0 * fbl[0], k1 * a1 * fbl[1]));
        st_shared_u32(sbase + L::OQ + sw128(t, col, 64), pack_bf16(q0 * a0 * fbl[0], q1 * a1 * fbl[1]));
        st_shared_u32(sbase + L::KE + sw128(t, col, 64), pack_bf16(k0 * e0 * fke[0], k1 * e1 * fke[1]));
        st_shared_u32(sbase + L::X + sw128(32 * I + r, col, 128), pack_bf16(k0 * a0, k1 * a1));
        st_shared_u32(sbase + L::X + sw128(32 * I + 16 + r, col, 128), pack_bf16(q0 * a0, q1 * a1));
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          uint32_t val;
          if (J == I)
            val = pack_bf16(k0 * ia0, k1 * ia1);
          else if (J > I)
            val = pack_bf16(k0 * e0 * fy[0][J], k1 * e1 * fy[1][J]);
          else
            val = 0u;
          st_shared_u32(sbase + L::Y + J * L::kYver + sw128(t, col, 64), val);
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();

    // the registers are free: start loading the next chunk
    if (ci + 1 < nchunks) prefetch(ci + 1);

    // ================= Gram^T: 4 versions =================
    if (tid == 0) {
      fence_after_sync();
      constexpr uint32_t id = idesc_bf16(128, 32, false, false);
#pragma unroll
      for (int I = 0; I < 4; ++I)
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tG + 32 * I, desc_kmajor(sbase + L::Y + I * L::kYver, 64, ks),
                   desc_kmajor(sbase + L::X, 128, ks, 32 * I), id, ks > 0);
      mma_commit(ctx.mbar);
    }
    wait_mma(ctx);

    // ---- Gram epilogue: lane j < 64 holds column j of L and A_Q ----
    if (tid < 64) {
      const int j = tid;
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        float v[32];
        tmem_ld32(tG + lane_base + 32 * I, v);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int i = 16 * I + r;
          sL[i * L::kLd + j] = (i > j) ? sBeta[i] * v[r] : 0.f;
          const float aq = (i >= j) ? v[16 + r] : 0.f;
          __nv_bfloat16 hq = __float2bfloat16_rn(aq);
          st_shared_u16(sbase + L::OQ + sw128(i, DK + j, 64), *reinterpret_cast<uint16_t*>(&hq));
        }
      }
    }
    __syncthreads();

    // ================= T = (I + L)^-1 (fp32) =================
    if (tid < 64) {  // diagonal 16 x 16 blocks, one column per thread
      const int I = tid >> 4, cc = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float s = (r == cc) ? 1.f : 0.f;
        if (r > cc) {
#pragma unroll
          for (int m = 0; m < r; ++m) s -= sL[(16 * I + r) * L::kLd + 16 * I + m] * x[m];
        }
        x[r] = (r >= cc) ? s : 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sT[(16 * I + r) * L::kLd + 16 * I + cc] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int I = 1; I < 4; ++I) {
      const int r = tid >> 3, jj = tid & 7;
      // R = L[I-block rows, 0:16I] * T[0:16I, 0:16I]
      for (int j = jj; j < 16 * I; j += 8) {
        float s = 0.f;
        for (int m = j; m < 16 * I; ++m) s += sL[(16 * I + r) * L::kLd + m] * sT[m * L::kLd + j];
        sR[r * L::kRd + j] = s;
      }
      __syncthreads();
      // T[I-block rows, 0:16I] = -T_II * R
      for (int j = jj; j < 16 * I; j += 8) {
        float s = 0.f;
        for (int m = 0; m <= r; ++m) s += sT[(16 * I + r) * L::kLd + 16 * I + m] * sR[m * L::kRd + j];
        sT[(16 * I + r) * L::kLd + j] = -s;
      }
      __syncthreads();
    }
    // T_beta = T Diag(beta) -> bf16 K-major [i][j]; also make sure V has landed
    cp_async_wait_all();
    {
      const int i = tid >> 1, j0 = 32 * (tid & 1);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ja = j0 + 8 * u + 2 * e, jb = ja + 1;
          const float xa = (ja <= i) ? sT[i * L::kLd + ja] * sBeta[ja] : 0.f;
          const float xb = (jb <= i) ? sT[i * L::kLd + jb] * sBeta[jb] : 0.f;
          w[e] = pack_bf16(xa, xb);
        }
        st_shared_v4(sbase + L::T2 + sw128(i, j0 + 8 * u, 64), w[0], w[1], w[2], w[3]);
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();

    // ================= W = T_beta K+ ,  U0 = T_beta V =================
    if (tid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t at = desc_kmajor(sbase + L::T2, 64, ks);
        mma_bf16(tG, at, desc_mnmajor(sbase + L::KP, 64, ks), idesc_bf16(128, DK, false, true), ks > 0);
        mma_bf16(tX, at, desc_mnmajor(sbase + L::VT, 64, ks), idesc_bf16(128, DV, false, true), ks > 0);
      }
      mma_commit(ctx.mbar);
    }
    wait_mma(ctx);
    __syncthreads();  // everyone is past the wait: V and K+ tiles are free
    if (*sFlag) break;
    if (ci + 1 < nchunks) prefetch_v(ci + 1);

    // ---- -W -> bf16 K-major rows 0..63 ----
    if (tid < 64) {
#pragma unroll
      for (int c0 = 0; c0 < DK; c0 += 32) {
        float v[32];
        tmem_ld32(tG + lane_base + c0, v);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(sbase + L::AW + sw128(tid, c0 + 8 * u, 64), pack_bf16(-v[8 * u], -v[8 * u + 1]),
                       pack_bf16(-v[8 * u + 2], -v[8 * u + 3]), pack_bf16(-v[8 * u + 4], -v[8 * u + 5]),
                       pack_bf16(-v[8 * u + 6], -v[8 * u + 7]));
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();

    // ================= serial step: U = U0 - W S =================
    if (tid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks)
        mma_bf16(tX, desc_kmajor(sbase + L::AW, 64, ks), desc_mnmajor(sbase + L::SB, DK, ks),
                 idesc_bf16(128, DV, false, true), 1u);
      mma_commit(ctx.mbar);
    }
    // meanwhile: S <- Diag(e^{G_C}) S in TMEM (rows are key channels)
    if (tid < DK) {
      const float pc = sP[tid];
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        float v[32];
        tmem_ld32(tS + lane_base + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= pc;
        tmem_st32(tS + lane_base + c0, v);
      }
    }
    wait_mma(ctx);

    // ---- U -> bf16 (MN-major [j][n]) ----
    if (tid < 64) {
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        float v[32];
        tmem_ld32(tX + lane_base + c0, v);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(sbase + L::KP + sw128(tid, c0 + 8 * u, 64), pack_bf16(v[8 * u], v[8 * u + 1]),
                       pack_bf16(v[8 * u + 2], v[8 * u + 3]), pack_bf16(v[8 * u + 4], v[8 * u + 5]),
                       pack_bf16(v[8 * u + 6], v[8 * u + 7]));
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();

    // ================= S += K_end^T U ;  O = [Q+ | A_Q] [S ; U] =================
    if (tid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tS, desc_mnmajor(sbase + L::KE, 64, ks), desc_mnmajor(sbase + L::KP, 64, ks),
                 idesc_bf16(128, DV, true, true), 1u);
#pragma unroll
      for (int ks = 0; ks < DK / 16 + 4; ++ks) {
        const int pnl = ks >> 2;
        const uint64_t ad =
            desc_sw128(sbase + L::OQ + (uint32_t)(pnl * 64 * 128) - 64 * 128 + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = ks < DK / 16 ? desc_mnmajor(sbase + L::SB, DK, ks)
                                         : desc_mnmajor(sbase + L::KP, 64, ks - DK / 16);
        mma_bf16(tX, ad, bd, idesc_bf16(128, DV, false, true), ks > 0);
      }
      mma_commit(ctx.mbar);
    }
    wait_mma(ctx);

    // ---- outputs (lanes 64..127) and the bf16 copy of the new state ----
    if (warp >= 2) {
      const int t = tid - 64;
      __nv_bfloat16* orow = og + ((int64_t)ci * kC + t) * a.out_st;
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        float v[32];
        tmem_ld32(tX + lane_base + c0, v);
        if (t < lc) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16(a.scale * v[8 * u], a.scale * v[8 * u + 1]);
            w.y = pack_bf16(a.scale * v[8 * u + 2], a.scale * v[8 * u + 3]);
            w.z = pack_bf16(a.scale * v[8 * u + 4], a.scale * v[8 * u + 5]);
            w.w = pack_bf16(a.scale * v[8 * u + 6], a.scale * v[8 * u + 7]);
            *reinterpret_cast<uint4*>(orow + c0 + 8 * u) = w;
          }
        }
      }
    }
    if (tid < DK) {
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        float v[32];
        tmem_ld32(tS + lane_base + c0, v);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(sbase + L::SB + sw128(tid, c0 + 8 * u, DK), pack_bf16(v[8 * u], v[8 * u + 1]),
                       pack_bf16(v[8 * u + 2], v[8 * u + 3]), pack_bf16(v[8 * u + 4], v[8 * u + 5]),
                       pack_bf16(v[8 * u + 6], v[8 * u + 7]));
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (*sFlag) break;
  }

  // ---- final state ----
  cp_async_wait_all();
  if (a.sT && tid < DK) {
    float* dst = a.sT + n * a.sT_sn + h * a.sT_sh + (int64_t)tid * DV;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float v[32];
      tmem_ld32(tS + lane_base + c0, v);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

template <int DK, int DV>
cudaError_t launch(const PrefillArgs& a, cudaStream_t s) {
  using L = Smem<DK, DV>;
  auto fn = kda_chunk_prefill_kernel<DK, DV>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  fn<<<dim3((unsigned)(a.N * a.H)), kThreads, L::kAlloc, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  if (!a.bf16) return cudaErrorInvalidValue;
  if (a.dk == 128 && a.dv == 128) return launch<128, 128>(a, s);
  if (a.dk == 128 && a.dv == 64) return launch<128, 64>(a, s);
  if (a.dk == 64 && a.dv == 128) return launch<64, 128>(a, s);
  if (a.dk == 64 && a.dv == 64) return launch<64, 64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
