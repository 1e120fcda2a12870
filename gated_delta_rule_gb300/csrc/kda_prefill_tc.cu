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
//     The column operand therefore exists in 4 versions, one per I; product I
//     covers all 128 rows [K; Q] and only its row block I is kept.
//   * K+ = K e^{G}, Q+ = Q e^{G}, K e^{G_C - G} are all <= 1.
//
// Tensor-core products (bf16 operands, fp32 accumulators in TMEM):
//   Gram (4 x [128 x 64 x d_k]), W / U0 (T_beta times [K+ | V]),
//   [U0 - W S] (the serial product with the bf16 copy of S),
//   S += K_end^T U, O = [Q+ | A_Q] [S ; U].
// The triangular inverse T: 16 x 16 diagonal blocks by fp32 forward
// substitution on the CUDA cores, then three block rows with warp-level
// tf32 MMAs (the blocks are 16 x 16, below the tcgen05 minimum M of 64).
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
  static constexpr int kLd = 68;  // fp32 row stride of L (16-byte rows, conflict-free tf32 loads)
  static constexpr int kTd = 72;  // fp32 row stride of T
  static constexpr int kRd = 56;  // fp32 row stride of the block-row workspace
  static constexpr int SL = 0;
  static constexpr int ST = SL + 64 * kLd * 4;
  static constexpr int SR = ST + 64 * kTd * 4;
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
  static constexpr int kParts = kThreads / (DK / 8);
  static constexpr int MBAR = CARRY + kParts * DK * 4;
  static constexpr int TSLOT = MBAR + 8;
  static constexpr int FLAG = TSLOT + 4;
  static constexpr int kTotal = FLAG + 4;
  static constexpr int kAlloc = kTotal + 1024;  // slack to align the base to 1024 bytes
  static_assert(kAlloc <= 232448, "shared memory budget");
  static constexpr uint32_t kTmemCols = 512;  // Gram 4 x 64, then U/O and S (DV each)
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

// 2^x on the special-function unit (relative error ~2^-22; results below
// 2^-126 flush to zero, which only drops contributions that small).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// D += A B on one warp: m16n8k8, tf32 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) kda_chunk_prefill_kernel(PrefillArgs a) {
  using L = Smem<DK, DV>;
  constexpr int OCT = DK / 8;            // channel octets
  constexpr int NPART = kThreads / OCT;  // token parts in the build
  constexpr int TPP = 64 / NPART;        // tokens per part (8 or 4)
  static_assert(16 % TPP == 0, "a part lies inside one 16-token sub-block");

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
  const int lane = tid & 31;
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
  const uint32_t tG = tmem;             // Gram (4 x 64 cols), then W (DK cols)
  const uint32_t tX = tmem + 256;       // U0 / U / O   (DV cols)
  const uint32_t tS = tmem + 256 + DV;  // fp32 state   (DV cols)
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

  // ---- per-thread build registers: channel octet `oct`, tokens [part*TPP, +TPP) ----
  const int oct = tid % OCT;
  const int part = tid / OCT;
  const int blk = (part * TPP) >> 4;  // this part's 16-token sub-block
  uint4 rk[TPP], rq[TPP];
  float4 rg[TPP][2];
  float rbeta = 0.f;

  auto chunk_len = [&](int ci) { return (int)(len - (int64_t)ci * kC < kC ? len - (int64_t)ci * kC : kC); };
  auto prefetch_kq = [&](int ci) {
    const int lc = chunk_len(ci);
#pragma unroll
    for (int i = 0; i < TPP; ++i) {
      const int t = part * TPP + i;
      const int64_t row = (int64_t)ci * kC + t;
      rk[i] = t < lc ? __ldg(reinterpret_cast<const uint4*>(kg + row * a.k.st) + oct) : make_uint4(0, 0, 0, 0);
      rq[i] = t < lc ? __ldg(reinterpret_cast<const uint4*>(qg + row * a.q.st) + oct) : make_uint4(0, 0, 0, 0);
    }
  };
  auto prefetch_g = [&](int ci) {
    const int lc = chunk_len(ci);
#pragma unroll
    for (int i = 0; i < TPP; ++i) {
      const int t = part * TPP + i;
      const int64_t row = (int64_t)ci * kC + t;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      rg[i][0] = t < lc ? __ldg(reinterpret_cast<const float4*>(gg + row * a.g.st) + 2 * oct) : z;
      rg[i][1] = t < lc ? __ldg(reinterpret_cast<const float4*>(gg + row * a.g.st) + 2 * oct + 1) : z;
    }
    rbeta = (tid < lc) ? __ldg(bg + ((int64_t)ci * kC + tid) * a.beta_st) : 0.f;
  };
  auto prefetch_v = [&](int ci) {
    const int lc = chunk_len(ci);
    constexpr int kVec = DV / 8;  // 16-byte vectors per row
#pragma unroll
    for (int it = 0; it < (64 * kVec) / kThreads; ++it) {
      const int idx = it * kThreads + tid;
      const int t = idx / kVec, cv = idx % kVec;
      const bool ok = t < lc;
      const __nv_bfloat16* src = ok ? vg + ((int64_t)ci * kC + t) * a.v.st + 8 * cv : vg;
      cp_async16(sbase + L::VT + sw128(t, 8 * cv, 64), src, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  if (nchunks > 0) {
    prefetch_kq(0);
    prefetch_g(0);
    prefetch_v(0);
  }

  for (int ci = 0; ci < nchunks; ++ci) {
    const int lc = chunk_len(ci);

    // ================= build: in-chunk scan and operand tiles =================
    // G (log2 units) for this thread's 8 channels and TPP tokens, then the carry
    // from the earlier parts of the chunk.
    float G[TPP][8];
    {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < TPP; ++i) {
        const float gv[8] = {rg[i][0].x, rg[i][0].y, rg[i][0].z, rg[i][0].w,
                             rg[i][1].x, rg[i][1].y, rg[i][1].z, rg[i][1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[e] = fmaf(gv[e], kLog2e, acc[e]);
          G[i][e] = acc[e];
        }
      }
      float4* cw = reinterpret_cast<float4*>(sCarry + part * DK + 8 * oct);
      cw[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      cw[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      if (tid < 64) sBeta[tid] = rbeta;
    }
    __syncthreads();
    {
      float off[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < part; ++q) {
        const float4* cr = reinterpret_cast<const float4*>(sCarry + q * DK + 8 * oct);
        const float4 x0 = cr[0], x1 = cr[1];
        off[0] += x0.x; off[1] += x0.y; off[2] += x0.z; off[3] += x0.w;
        off[4] += x1.x; off[5] += x1.y; off[6] += x1.z; off[7] += x1.w;
      }
#pragma unroll
      for (int i = 0; i < TPP; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) G[i][e] += off[e];
      float4* b0 = reinterpret_cast<float4*>(sBnd + 8 * oct);
      if (part == 0) {
        b0[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        b0[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (((part + 1) * TPP) % 16 == 0) {  // this part ends a sub-block: publish its boundary
        const int kb = ((part + 1) * TPP) >> 4;
        float4* bw = reinterpret_cast<float4*>(sBnd + kb * DK + 8 * oct);
        bw[0] = make_float4(G[TPP - 1][0], G[TPP - 1][1], G[TPP - 1][2], G[TPP - 1][3]);
        bw[1] = make_float4(G[TPP - 1][4], G[TPP - 1][5], G[TPP - 1][6], G[TPP - 1][7]);
        if (kb == 4) {
          float4* pw = reinterpret_cast<float4*>(sP + 8 * oct);
          pw[0] = make_float4(exp2f(G[TPP - 1][0]), exp2f(G[TPP - 1][1]), exp2f(G[TPP - 1][2]), exp2f(G[TPP - 1][3]));
          pw[1] = make_float4(exp2f(G[TPP - 1][4]), exp2f(G[TPP - 1][5]), exp2f(G[TPP - 1][6]), exp2f(G[TPP - 1][7]));
        }
      }
    }
    __syncthreads();
    {
      // per-channel factors of this thread's sub-block I = blk (log2 units):
      //   bl = G before the block, en = G at its end, pe = G at the chunk end.
      //   fbl = 2^bl, hI = 2^(en - bl), hk = hI 2^(pe - en), f2/f3 = 2^(G at the
      //   start of block blk+2 / blk+3 - en) (the version for block blk+1 needs none).
      float fbl[8], hI[8], hk[8], f2[8], f3[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = 8 * oct + e;
        const float bl = sBnd[blk * DK + c];
        const float en = sBnd[(blk + 1) * DK + c];
        fbl[e] = ex2(bl);
        hI[e] = ex2(en - bl);
        hk[e] = hI[e] * ex2(sBnd[4 * DK + c] - en);
        f2[e] = blk + 2 <= 3 ? ex2(sBnd[min(blk + 2, 4) * DK + c] - en) : 0.f;
        f3[e] = blk + 3 <= 3 ? ex2(sBnd[min(blk + 3, 4) * DK + c] - en) : 0.f;
#pragma unroll
        for (int i = 0; i < TPP; ++i) G[i][e] -= bl;  // G now relative to the block start
      }
      const int col = 8 * oct;
      auto st8 = [&](uint32_t addr, const float* x) {
        st_shared_v4(addr, pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                     pack_bf16(x[6], x[7]));
      };
#pragma unroll
      for (int i = 0; i < TPP; ++i) {
        const int t = part * TPP + i;
        const uint32_t kw[4] = {rk[i].x, rk[i].y, rk[i].z, rk[i].w};
        const uint32_t qw[4] = {rq[i].x, rq[i].y, rq[i].z, rq[i].w};
        float av[8], ia[8], x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          av[e] = ex2(G[i][e]);
          ia[e] = ex2(-G[i][e]);
        }
        // rows of the Gram (block-local) and K+ = K e^{G}
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = ((e & 1) ? bf_hi(kw[e >> 1]) : bf_lo(kw[e >> 1])) * av[e];
        st8(sbase + L::X + sw128(t, col, 128), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= fbl[e];
        st8(sbase + L::KP + sw128(t, col, 64), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = ((e & 1) ? bf_hi(qw[e >> 1]) : bf_lo(qw[e >> 1])) * av[e];
        st8(sbase + L::X + sw128(64 + t, col, 128), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= fbl[e];
        st8(sbase + L::OQ + sw128(t, col, 64), x);
        // column versions: own block k e^{-G}, later blocks k e^{en - G} (times f2, f3)
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = ((e & 1) ? bf_hi(kw[e >> 1]) : bf_lo(kw[e >> 1])) * ia[e];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = y[e] * hk[e];
        st8(sbase + L::KE + sw128(t, col, 64), x);
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          const uint32_t addr = sbase + L::Y + J * L::kYver + sw128(t, col, 64);
          if (J < blk) {
            st_shared_v4(addr, 0u, 0u, 0u, 0u);
          } else if (J == blk) {
            st8(addr, y);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              x[e] = y[e] * hI[e] * (J == blk + 1 ? 1.f : (J == blk + 2 ? f2[e] : f3[e]));
            st8(addr, x);
          }
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();

    // ================= Gram: row block I uses column version I =================
    if (tid == 0) {
      fence_after_sync();
      constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int I = 0; I < 4; ++I)
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tG + 64 * I, desc_kmajor(sbase + L::X, 128, ks),
                   desc_kmajor(sbase + L::Y + I * L::kYver, 64, ks), id, ks > 0);
      mma_commit(ctx.mbar);
    }
    // the k/q registers are free: start loading the next chunk while the MMAs run
    if (ci + 1 < nchunks) prefetch_kq(ci + 1);
    wait_mma(ctx);

    // ---- Gram epilogue: lane i < 64 -> row i of L (fp32), lane 64 + i -> row i of A_Q (bf16) ----
    {
      const int i = tid & 63;
      const int myblk = i >> 4;
      const int b0 = (warp & 1) * 2;  // the two row blocks this warp's lanes fall in
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(tG + lane_base + 64 * (b0 + bb) + 32 * half, v);
          if (myblk == b0 + bb) {
            const int j0 = 32 * half;
            if (tid < 64) {
              const float bi = sBeta[i];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                float4 w;
                w.x = (j0 + 4 * u + 0 < i) ? bi * v[4 * u + 0] : 0.f;
                w.y = (j0 + 4 * u + 1 < i) ? bi * v[4 * u + 1] : 0.f;
                w.z = (j0 + 4 * u + 2 < i) ? bi * v[4 * u + 2] : 0.f;
                w.w = (j0 + 4 * u + 3 < i) ? bi * v[4 * u + 3] : 0.f;
                *reinterpret_cast<float4*>(sL + i * L::kLd + j0 + 4 * u) = w;
              }
            } else {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (j0 + 8 * u + e <= i) ? v[8 * u + e] : 0.f;
                st_shared_v4(sbase + L::OQ + sw128(i, DK + j0 + 8 * u, 64), pack_bf16(x[0], x[1]),
                             pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
              }
            }
          }
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
      for (int r = 0; r < 16; ++r) sT[(16 * I + r) * L::kTd + 16 * I + cc] = x[r];
    }
    __syncthreads();
    // block rows I = 1..3 on the warp-level tensor cores (tf32, fp32 accumulate):
    //   R = L[I, 0:16I] T[0:16I, 0:16I] ;  T[I, 0:16I] = -T_II R
    // Each warp owns whole 8-column tiles, so R stays within the warp.
    {
      const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int I = 1; I < 4; ++I) {
        for (int nt = warp; nt < 2 * I; nt += 4) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int ks = 2 * (nt >> 1); ks < 2 * I; ++ks) {
            const int k0 = 8 * ks;
            const float* l0 = sL + (16 * I + gq) * L::kLd + k0 + tq;
            const float* l1 = l0 + 8 * L::kLd;
            const uint32_t af[4] = {to_tf32(l0[0]), to_tf32(l1[0]), to_tf32(l0[4]), to_tf32(l1[4])};
            const uint32_t bf[2] = {to_tf32(sT[(k0 + tq) * L::kTd + 8 * nt + gq]),
                                    to_tf32(sT[(k0 + tq + 4) * L::kTd + 8 * nt + gq])};
            mma_tf32(acc, af, bf);
          }
          sR[gq * L::kRd + 8 * nt + 2 * tq] = acc[0];
          sR[gq * L::kRd + 8 * nt + 2 * tq + 1] = acc[1];
          sR[(gq + 8) * L::kRd + 8 * nt + 2 * tq] = acc[2];
          sR[(gq + 8) * L::kRd + 8 * nt + 2 * tq + 1] = acc[3];
          __syncwarp();
          float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const int k0 = 8 * ks;
            const float* t0 = sT + (16 * I + gq) * L::kTd + 16 * I + k0 + tq;
            const float* t1 = t0 + 8 * L::kTd;
            const uint32_t af[4] = {to_tf32(t0[0]), to_tf32(t1[0]), to_tf32(t0[4]), to_tf32(t1[4])};
            const uint32_t bf[2] = {to_tf32(sR[(k0 + tq) * L::kRd + 8 * nt + gq]),
                                    to_tf32(sR[(k0 + tq + 4) * L::kRd + 8 * nt + gq])};
            mma_tf32(acc2, af, bf);
          }
          float* d0 = sT + (16 * I + gq) * L::kTd + 8 * nt + 2 * tq;
          float* d1 = d0 + 8 * L::kTd;
          d0[0] = -acc2[0];
          d0[1] = -acc2[1];
          d1[0] = -acc2[2];
          d1[1] = -acc2[3];
        }
        __syncthreads();
      }
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
          const float xa = (ja <= i) ? sT[i * L::kTd + ja] * sBeta[ja] : 0.f;
          const float xb = (jb <= i) ? sT[i * L::kTd + jb] * sBeta[jb] : 0.f;
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
    if (ci + 1 < nchunks) prefetch_g(ci + 1);
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
