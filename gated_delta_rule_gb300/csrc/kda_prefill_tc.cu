// Chunked KDA prefill on the sm_100-family tensor cores (tcgen05 + TMEM).
//
// The chunked form of "尝试对Kimi KDA的数学推导&算子实现分析" (hjcheng0602.cn/blog/kdd),
// per chunk of C = 64 tokens, written with U = (I + L)^-1 B_beta (V - K+ S):
//
//   G_t   = sum_{r <= t} g_r inside the chunk                          (eq. 9)
//   L     = StrictTril(B_beta K+ K-^T)                                  (eq. 51)
//   A_Q   = Tril(Q+ K-^T)   (inclusive; the read-out sums j <= t)       (eq. 57)
//   T     = (I + L)^-1                                                  (eq. 27)
//   W     = T B_beta K+                         (S-independent)         (eq. 52)
//   U     = T B_beta V - W S                                            (eq. 52)
//   O     = scale (Q+ S + A_Q U)                                        (eq. 63)
//   S'    = Diag(e^{G_C}) S + (K e^{G_C - G})^T U                       (eqs. 64-66)
//
// Two kernels, like the K1 / K2 split the page describes for FlashKDA, laid
// out for sm_103a:
//   * kda_chunk_prep_kernel: every (chunk, head) on its own, persistent CTAs,
//     two per SM.  It forms the in-chunk cumulative log-decay, the operand
//     tiles, the Gram products (tcgen05), the triangular inverse (CUDA cores +
//     warp-level tf32 MMA) and W (tcgen05), and writes one "chunk record" of
//     ready-to-use swizzled bf16 tiles -- T B_beta, [-W ; Q+], A_Q,
//     (K e^{G_C - G})^T -- plus e^{G_C} to a workspace.
//   * kda_chunk_serial_kernel: one CTA per (sequence, head) keeps the fp32 state
//     in TMEM and walks the chunks in order, with warp roles: a producer warp
//     (record by bulk copy, V by cp.async, one chunk ahead), an MMA warp and
//     four TMEM <-> memory warps.  Each chunk costs three tcgen05 products:
//     [U ; Q+ S] = [T_beta | -W ; 0 | Q+] [V ; S], then S += K_end^T U on the
//     state chain and O += A_Q U off it; the U/O accumulator is double-buffered
//     in TMEM so the output epilogue overlaps the next chunk.
//
// Exponents are only ever formed as differences that stay inside a 16-token
// sub-block or decay toward the later token, so nothing overflows for
// g in [-5, 0] (the lower-bounded decay of "Kimi K3 技术报告解读"
// (marsggbo.github.io) §3.5: a 16-token cumulative log-decay stays in (-80, 0]):
//   * Gram blocks use, for output rows in sub-block I, the reference G at the
//     start of sub-block I: rows K_i e^{G_i - G_{16I-1}} (<= 1) and columns
//     K_j e^{G_{16I-1} - G_j} (<= 1 for earlier sub-blocks, < e^80 inside I).
//     The column operand exists in 4 versions (16, 32, 48, 64 rows); product I
//     covers all 128 rows [K; Q] and only its row block I is kept.
//   * K+ = K e^{G}, Q+ = Q e^{G}, K e^{G_C - G} are all <= 1.
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

// One chunk record (per chunk and head), byte offsets.  Tiles are stored exactly
// as they sit in shared memory, so one bulk copy moves the whole record.
template <int DK>
struct Rec {
  static constexpr int T2 = 0;                      // T Diag(beta): 64 x 64, K-major
  static constexpr int WQ = T2 + 64 * 64 * 2;       // [-W ; Q+]: 128 x DK, K-major
  static constexpr int AQ = WQ + 128 * DK * 2;      // A_Q: 64 x 64, K-major
  static constexpr int KE = AQ + 64 * 64 * 2;       // (K e^{G_C - G})^T: DK x 64, K-major
  static constexpr int P = KE + 64 * DK * 2;        // e^{G_C}: DK fp32
  static constexpr int kBytes = align1k(P + DK * 4);
};

// Gram column versions: version I has 16 (I + 1) rows.
__host__ __device__ constexpr int yrows(int I) { return 16 * (I + 1); }
__host__ __device__ constexpr int yoff_rows(int I) { return 8 * I * (I + 1); }  // rows before version I

template <int DK>
struct PrepSmem {
  static constexpr int X = 0;                          // 128 rows [K; Q] x DK, K-major
  static constexpr int Y = X + 128 * DK * 2;           // versions 0..3, 160 rows x DK, K-major
  static constexpr int kGram = Y + 160 * DK * 2;
  static constexpr int kLd = 68;  // fp32 row stride of L (16-byte rows, conflict-free tf32 loads)
  static constexpr int kTd = 72;  // fp32 row stride of T
  static constexpr int kRd = 56;  // fp32 row stride of the block-row workspace
  static constexpr int SL = 0;
  static constexpr int ST = SL + 64 * kLd * 4;
  static constexpr int SR = ST + 64 * kTd * 4;
  static constexpr int T2 = align1k(SR + 16 * kRd * 4);  // 64 x 64 bf16 (+ an 8K window)
  static constexpr int kSolve = T2 + 2 * 64 * 64 * 2;
  static constexpr int kG = kGram > kSolve ? kGram : kSolve;
  static constexpr int KP = align1k(kG);  // K+ : [64 tokens][DK], MN-major
  static constexpr int BETA = KP + 64 * DK * 2;
  static constexpr int BND = BETA + 64 * 4;  // 5 x DK fp32 (log2 units)
  static constexpr int kParts = kThreads / (DK / 8);
  static constexpr int CARRY = BND + 5 * DK * 4;
  static constexpr int MBAR = CARRY + kParts * DK * 4;
  static constexpr int TSLOT = MBAR + 8;
  static constexpr int FLAG = TSLOT + 4;
  static constexpr int kAlloc = FLAG + 4 + 1024;
  static_assert(2 * (kAlloc + 1024) <= 233472, "two prep CTAs per SM");
  static constexpr uint32_t kTmemCols = 256;  // Gram 160 cols, then W (DK cols)
};

template <int DK, int DV>
struct SerialSmem {
  // a record buffer holds [T2 | zero tile | rest of the record]: the zero tile is
  // the lower half of T2's M = 128 window
  static constexpr int kRecBuf = align1k(Rec<DK>::kBytes + 64 * 64 * 2);
  static constexpr int REC = 0;                          // two record buffers
  static constexpr int VT = REC + 2 * kRecBuf;           // two V chunks [64][DV] MN-major (U reuses)
  static constexpr int SB = VT + 2 * 64 * DV * 2;        // bf16 S, [DK][DV] MN-major
  static constexpr int OSTG = SB + DK * DV * 2;          // output staging: 2 warps x 32 rows x 144 B
  static constexpr int MBAR = OSTG + 2 * 32 * 144;       // mma_a, mma_s, rec0/1, free0/1, orel0/1
  static constexpr int TSLOT = MBAR + 64;
  static constexpr int FLAG = TSLOT + 4;
  static constexpr int kAlloc = FLAG + 4 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget");
  static constexpr uint32_t kTmemCols = 3 * DV <= 256 ? 256 : 512;  // U/O x2 and S
};

struct Split {
  unsigned char* rec;  // records: [chunk index][head][Rec bytes]
  const int* off;      // first chunk index of each sequence ([N + 1]); null for fixed length
  int total;           // chunk indices allocated (an upper bound with varlen)
  int nck;             // chunks per sequence when fixed length
};

struct Range {
  int64_t brow, tok0;
  int len;
};

// Token range of sequence n, clamped exactly as every kernel here clamps it.
__device__ __forceinline__ Range seq_range(const PrefillArgs& a, int n) {
  Range r{n, 0, a.T};
  if (a.cu_seqlens) {
    const int c0 = min(max(__ldg(a.cu_seqlens + n), 0), a.T);
    const int c1 = min(max(__ldg(a.cu_seqlens + n + 1), c0), a.T);
    r.brow = 0;
    r.tok0 = c0;
    r.len = c1 - c0;
  }
  return r;
}

__device__ __forceinline__ int first_chunk(const Split& sp, int n) {
  return sp.off ? __ldg(sp.off + n) : n * sp.nck;
}
__device__ __forceinline__ int num_chunks(const Split& sp, int n) {
  return sp.off ? __ldg(sp.off + n + 1) - __ldg(sp.off + n) : sp.nck;
}

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


// ---------------------------------------------------------------------------
// prep: one chunk of one head per iteration; persistent CTAs
template <int DK>
__global__ void __launch_bounds__(kThreads, 2) kda_chunk_prep_kernel(PrefillArgs a, Split sp) {
  using L = PrepSmem<DK>;
  using R = Rec<DK>;
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
  float* sBnd = reinterpret_cast<float*>(smem + L::BND);
  float* sCarry = reinterpret_cast<float*>(smem + L::CARRY);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + L::FLAG);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

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
  Ctx ctx{sbase + L::MBAR, 0u, sFlag, a.err};

  const int oct = tid % OCT;
  const int part = tid / OCT;
  const int blk = (part * TPP) >> 4;  // this part's 16-token sub-block
  const int nitems = sp.total * a.H;
  const int nseq_chunks = sp.off ? __ldg(sp.off + a.N) : sp.total;

  // item w -> (sequence n, chunk ci, head h); valid == false past the last chunk
  struct Item {
    bool valid;
    int n, h, lc;
    int64_t brow, row0;  // batch row and first token row of the chunk
    int64_t rec;         // record index
  };
  auto item = [&](int w) {
    Item it{false, 0, 0, 0, 0, 0, 0};
    if (w >= nitems) return it;
    const int g = w / a.H;
    it.h = w - g * a.H;
    if (g >= nseq_chunks) return it;
    int n;
    if (sp.off) {  // largest n with off[n] <= g
      int lo = 0, hi = a.N - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(sp.off + mid) <= g) lo = mid; else hi = mid - 1;
      }
      n = lo;
    } else {
      n = g / sp.nck;
    }
    const int ci = g - first_chunk(sp, n);
    const Range r = seq_range(a, n);
    it.valid = true;
    it.n = n;
    it.brow = r.brow;
    it.row0 = r.tok0 + (int64_t)ci * kC;
    it.lc = min(kC, r.len - ci * kC);
    it.rec = (int64_t)g * a.H + it.h;
    return it;
  };

  uint4 rk[TPP], rq[TPP];
  float4 rg[TPP][2];
  float rbeta = 0.f;
  auto load_kq = [&](const Item& it) {
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(a.k.ptr) + it.brow * a.k.sb + it.h * a.k.sh;
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q.ptr) + it.brow * a.q.sb + it.h * a.q.sh;
#pragma unroll
    for (int i = 0; i < TPP; ++i) {
      const int t = part * TPP + i;
      const bool ok = it.valid && t < it.lc;
      const int64_t row = it.row0 + t;
      rk[i] = ok ? __ldg(reinterpret_cast<const uint4*>(kb + row * a.k.st) + oct) : make_uint4(0, 0, 0, 0);
      rq[i] = ok ? __ldg(reinterpret_cast<const uint4*>(qb + row * a.q.st) + oct) : make_uint4(0, 0, 0, 0);
    }
  };
  auto load_g = [&](const Item& it) {
    const float* gb = static_cast<const float*>(a.g.ptr) + it.brow * a.g.sb + it.h * a.g.sh;
#pragma unroll
    for (int i = 0; i < TPP; ++i) {
      const int t = part * TPP + i;
      const bool ok = it.valid && t < it.lc;
      const int64_t row = it.row0 + t;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      rg[i][0] = ok ? __ldg(reinterpret_cast<const float4*>(gb + row * a.g.st) + 2 * oct) : z;
      rg[i][1] = ok ? __ldg(reinterpret_cast<const float4*>(gb + row * a.g.st) + 2 * oct + 1) : z;
    }
    const float* bb = a.beta + it.brow * a.beta_sb + it.h * a.beta_sh;
    rbeta = (it.valid && tid < it.lc) ? __ldg(bb + (it.row0 + tid) * a.beta_st) : 0.f;
  };

  Item cur = item(blockIdx.x);
  load_kq(cur);
  load_g(cur);

  for (int w = blockIdx.x; w < nitems; w += gridDim.x) {
    const Item nxt = item(w + gridDim.x);
    if (cur.valid) {
      unsigned char* rec = sp.rec + cur.rec * R::kBytes;

      // ================= scan: G (log2 units) for 8 channels x TPP tokens =================
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
        if (part == 0) {
          float4* b0 = reinterpret_cast<float4*>(sBnd + 8 * oct);
          b0[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          b0[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (((part + 1) * TPP) % 16 == 0) {  // this part ends a sub-block: publish its boundary
          const int kb = ((part + 1) * TPP) >> 4;
          float4* bw = reinterpret_cast<float4*>(sBnd + kb * DK + 8 * oct);
          bw[0] = make_float4(G[TPP - 1][0], G[TPP - 1][1], G[TPP - 1][2], G[TPP - 1][3]);
          bw[1] = make_float4(G[TPP - 1][4], G[TPP - 1][5], G[TPP - 1][6], G[TPP - 1][7]);
          if (kb == 4) {  // the chunk's state decay e^{G_C}
            float4* pw = reinterpret_cast<float4*>(rec + R::P + 32 * oct);
            pw[0] = make_float4(exp2f(G[TPP - 1][0]), exp2f(G[TPP - 1][1]), exp2f(G[TPP - 1][2]),
                                exp2f(G[TPP - 1][3]));
            pw[1] = make_float4(exp2f(G[TPP - 1][4]), exp2f(G[TPP - 1][5]), exp2f(G[TPP - 1][6]),
                                exp2f(G[TPP - 1][7]));
          }
        }
      }
      __syncthreads();

      // ================= build: operand tiles =================
      {
        // per-channel factors of sub-block blk (log2 units): bl = G before the
        // block, en = G at its end, pe = G at the chunk end.  fbl = 2^bl,
        // hI = 2^(en - bl), hk = hI 2^(pe - en), f2 / f3 = 2^(G at the start of
        // block blk+2 / blk+3 - en).
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
        auto pack8 = [&](const float* x) {
          return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                            pack_bf16(x[6], x[7]));
        };
        auto st8 = [&](uint32_t addr, const float* x) {
          const uint4 u = pack8(x);
          st_shared_v4(addr, u.x, u.y, u.z, u.w);
        };
        // K_end^T is stored K-major ([channel][token]): this thread's 8 x TPP block,
        // packed in token pairs, is written once after the token loop
        uint32_t ket[8][TPP / 2];
        float ke_even[8];
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
          // Gram rows (block-local) and K+ = K e^{G}
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = ((e & 1) ? bf_hi(kw[e >> 1]) : bf_lo(kw[e >> 1])) * av[e];
          st8(sbase + L::X + sw128(t, col, 128), x);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= fbl[e];
          st8(sbase + L::KP + sw128(t, col, 64), x);
          // Gram rows of q and Q+ = Q e^{G} (record)
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = ((e & 1) ? bf_hi(qw[e >> 1]) : bf_lo(qw[e >> 1])) * av[e];
          st8(sbase + L::X + sw128(64 + t, col, 128), x);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= fbl[e];
          *reinterpret_cast<uint4*>(rec + R::WQ + sw128(64 + t, col, 128)) = pack8(x);
          // column versions: own block k e^{-G}; later blocks k e^{en - G} (x f2, f3); and K_end
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = ((e & 1) ? bf_hi(kw[e >> 1]) : bf_lo(kw[e >> 1])) * ia[e];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float ke = y[e] * hk[e];
            if (i & 1)
              ket[e][i >> 1] = pack_bf16(ke_even[e], ke);
            else
              ke_even[e] = ke;
          }
#pragma unroll
          for (int J = 0; J < 4; ++J) {
            if (J < blk) continue;
            const uint32_t addr = sbase + L::Y + yoff_rows(J) * DK * 2 + sw128(t, col, yrows(J));
            if (J == blk) {
              st8(addr, y);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                x[e] = y[e] * hI[e] * (J == blk + 1 ? 1.f : (J == blk + 2 ? f2[e] : f3[e]));
              st8(addr, x);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          unsigned char* dst = rec + R::KE + sw128(col + e, part * TPP, DK);
          if constexpr (TPP == 8)
            *reinterpret_cast<uint4*>(dst) = make_uint4(ket[e][0], ket[e][1], ket[e][2], ket[e][3]);
          else
            *reinterpret_cast<uint2*>(dst) = make_uint2(ket[e][0], ket[e][1]);
        }
      }
      fence_async_smem();
      fence_before_sync();
      __syncthreads();

      // ================= Gram: row block I against column version I =================
      if (tid == 0) {
        fence_after_sync();
#pragma unroll
        for (int I = 0; I < 4; ++I)
#pragma unroll
          for (int ks = 0; ks < DK / 16; ++ks)
            mma_bf16(tmem + yoff_rows(I), desc_kmajor(sbase + L::X, 128, ks),
                     desc_kmajor(sbase + L::Y + yoff_rows(I) * DK * 2, yrows(I), ks),
                     idesc_bf16(128, yrows(I), false, false), ks > 0);
        mma_commit(ctx.mbar);
      }
      // the k/q registers are free: start loading the next item while the MMAs run
      load_kq(nxt);
      wait_mma(ctx);

      // ---- Gram epilogue: lane i < 64 -> row i of L (fp32); lane 64 + i -> row i of A_Q ----
      {
        const int i = tid & 63;
        const int myblk = i >> 4;
        const int b0 = (warp & 1) * 2;  // this warp's lanes fall in row blocks b0, b0 + 1
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int b = b0 + bb;
          for (int pc = 0; pc <= b; ++pc) {  // 16-column pieces of version b
            float v[16];
            tmem_ld16(tmem + lane_base + yoff_rows(b) + 16 * pc, v);
            if (myblk == b) {
              const int j0 = 16 * pc;
              if (tid < 64) {
                const float bi = sBeta[i];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  float4 f;
                  f.x = (j0 + 4 * u + 0 < i) ? bi * v[4 * u + 0] : 0.f;
                  f.y = (j0 + 4 * u + 1 < i) ? bi * v[4 * u + 1] : 0.f;
                  f.z = (j0 + 4 * u + 2 < i) ? bi * v[4 * u + 2] : 0.f;
                  f.w = (j0 + 4 * u + 3 < i) ? bi * v[4 * u + 3] : 0.f;
                  *reinterpret_cast<float4*>(sL + i * L::kLd + j0 + 4 * u) = f;
                }
              } else {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  float x[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) x[e] = (j0 + 8 * u + e <= i) ? v[8 * u + e] : 0.f;
                  *reinterpret_cast<uint4*>(rec + R::AQ + sw128(i, j0 + 8 * u, 64)) =
                      make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                 pack_bf16(x[6], x[7]));
                }
              }
            }
          }
        }
        if (tid >= 64) {  // A_Q columns past this row's sub-block are zero
          for (int j0 = 16 * (myblk + 1); j0 < 64; j0 += 8)
            *reinterpret_cast<uint4*>(rec + R::AQ + sw128(i, j0, 64)) = make_uint4(0, 0, 0, 0);
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
      // T_beta = T Diag(beta) -> bf16 K-major [i][j], into shared memory and the record
      {
        const int i = tid >> 1, j0 = 32 * (tid & 1);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ja = j0 + 8 * u + 2 * e, jb = ja + 1;
            const float xa = (ja <= i) ? sT[i * L::kTd + ja] * sBeta[ja] : 0.f;
            const float xb = (jb <= i) ? sT[i * L::kTd + jb] * sBeta[jb] : 0.f;
            wv[e] = pack_bf16(xa, xb);
          }
          const uint32_t off = sw128(i, j0 + 8 * u, 64);
          st_shared_v4(sbase + L::T2 + off, wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(rec + R::T2 + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
      fence_async_smem();
      fence_before_sync();
      __syncthreads();

      // ================= W = T_beta K+ =================
      if (tid == 0) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem, desc_kmajor(sbase + L::T2, 64, ks), desc_mnmajor(sbase + L::KP, 64, ks),
                   idesc_bf16(128, DK, false, true), ks > 0);
        mma_commit(ctx.mbar);
      }
      load_g(nxt);
      wait_mma(ctx);
      // ---- -W -> record (bf16 K-major rows 0..63) ----
      if (tid < 64) {
#pragma unroll
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float v[32];
          tmem_ld32(tmem + lane_base + c0, v);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(rec + R::WQ + sw128(tid, c0 + 8 * u, 128)) =
                make_uint4(pack_bf16(-v[8 * u], -v[8 * u + 1]), pack_bf16(-v[8 * u + 2], -v[8 * u + 3]),
                           pack_bf16(-v[8 * u + 4], -v[8 * u + 5]), pack_bf16(-v[8 * u + 6], -v[8 * u + 7]));
        }
      }
      fence_before_sync();
      __syncthreads();
      if (*sFlag) break;
    } else {
      load_kq(nxt);
      load_g(nxt);
    }
    cur = nxt;
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------
// serial: one (sequence, head) per CTA, fp32 state in TMEM.
// Warps 0-3 move data between TMEM and shared / global memory, warp 4 issues the
// tensor-core products, warp 5 loads chunk records (bulk copy) and V (cp.async);
// both kinds of copy complete on the record buffer's mbarrier.  Hand-offs:
//   bar 1 (160): bf16 copy of the state entering the chunk is in shared memory
//   bar 2 (160): the TMEM state is decayed and U is in shared memory
//   mbarriers  : MMA completion (a: U / Q+S, s: state), records (plus V)
//                landed, a buffer's chunk finished (output ready, buffers
//                free), and orel[b]: warps 2-3 have read the output of buffer
//                b's chunk out of TMEM (64 arrivals), so the chunk two later may
//                write it.  (Per buffer, and an mbarrier rather than a named
//                barrier: warps 2-3 may arrive for the next chunk before the MMA
//                warp has waited for this one.)  Every mbarrier here is waited
//                on by a role that the barrier's next phase depends on, so no
//                waiter can fall two phases behind.
constexpr int kSerialThreads = 192;

template <int DK, int DV>
__global__ void __launch_bounds__(kSerialThreads, 1) kda_chunk_serial_kernel(PrefillArgs a, Split sp) {
  using L = SerialSmem<DK, DV>;
  using R = Rec<DK>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + L::FLAG);
  const uint32_t mbar_a = sbase + L::MBAR, mbar_s = mbar_a + 8;
  const uint32_t mbar_rec0 = mbar_a + 16;   // record (+ V) of buffer b landed
  const uint32_t mbar_free0 = mbar_a + 32;  // buffer b's chunk has finished its last product
  const uint32_t mbar_orel0 = mbar_a + 48;  // buffer b's output has been read out of TMEM
  constexpr int kT2 = 64 * 64 * 2;  // T2 tile bytes; the rest of a record lands after the zero tile

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const int n = blockIdx.x / a.H;
  const int h = blockIdx.x - n * a.H;
  const Range rg = seq_range(a, n);
  const int nch = min(num_chunks(sp, n), (rg.len + kC - 1) / kC);
  const int64_t rec0 = (int64_t)first_chunk(sp, n) * a.H + h;  // record of chunk ci: rec0 + ci * H

  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v.ptr) + rg.brow * a.v.sb + rg.tok0 * a.v.st + h * a.v.sh;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + rg.brow * a.out_sb + rg.tok0 * a.out_st + h * a.out_sh;

  if (tid == 0) {
    mbar_init(mbar_a, 1);
    mbar_init(mbar_s, 1);
    mbar_init(mbar_rec0, 33);  // producer lane 0's expect_tx arrival + 32 cp.async arrivals
    mbar_init(mbar_rec0 + 8, 33);
    mbar_init(mbar_free0, 1);
    mbar_init(mbar_free0 + 8, 1);
    mbar_init(mbar_orel0, 64);  // every thread of warps 2-3
    mbar_init(mbar_orel0 + 8, 64);
    fence_mbar_init();
    *sFlag = 0;
  }
  for (int i = tid; i < 2 * kT2 / 16; i += kSerialThreads) {  // zero tiles below each T2 buffer
    const int b = i / (kT2 / 16), o = i % (kT2 / 16);
    st_shared_v4(sbase + L::REC + b * L::kRecBuf + kT2 + 16 * o, 0u, 0u, 0u, 0u);
  }
  if (warp == 0) tmem_alloc(sbase + L::TSLOT, L::kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);
  const uint32_t tS = tmem + 2 * DV;  // fp32 state (DV cols); U/O buffers at 0 and DV
  auto tX = [&](int b) { return tmem + (uint32_t)(b * DV); };
  // bounded wait; after any timeout every later wait returns at once so all roles finish
  auto wait = [&](uint32_t mbar, uint32_t parity) {
    if (!*sFlag && !mbar_wait(mbar, parity)) {
      atomicOr(a.err, kErrTimeout);
      *sFlag = 1;
    }
    fence_after_sync();
  };

  if (tid < DK) {  // lane c holds state row c: TMEM <- S0, shared <- bf16(S0)
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
  fence_async_smem();
  fence_before_sync();
  __syncthreads();

  if (warp == 5) {
    // ======================= producer warp =======================
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      if (ci >= 2) wait(mbar_free0 + 8 * b, (uint32_t)(((ci - 2) >> 1) & 1));  // chunk ci - 2 is done
      const uint32_t dst = sbase + L::REC + b * L::kRecBuf;
      const uint32_t mb = mbar_rec0 + 8 * b;
      if (lane == 0) {
        const unsigned char* src = sp.rec + (rec0 + (int64_t)ci * a.H) * R::kBytes;
        mbar_arrive_expect_tx(mb, R::kBytes);
        bulk_g2s(dst, src, kT2, mb);
        bulk_g2s(dst + 2 * kT2, src + kT2, R::kBytes - kT2, mb);
      }
      const int lc = min(kC, rg.len - ci * kC);
      constexpr int kVec = DV / 8;
#pragma unroll 4
      for (int idx = lane; idx < 64 * kVec; idx += 32) {
        const int t = idx / kVec, cv = idx % kVec;
        const bool ok = t < lc;
        const __nv_bfloat16* src = ok ? vg + ((int64_t)ci * kC + t) * a.v.st + 8 * cv : vg;
        cp_async16(sbase + L::VT + b * 64 * DV * 2 + sw128(t, 8 * cv, 64), src, ok ? 16u : 0u);
      }
      cp_async_mbar_arrive(mb);
    }
    cp_async_wait_all();
  } else if (warp == 4) {
    // ======================= MMA warp =======================
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      const uint32_t rec = sbase + L::REC + b * L::kRecBuf;  // T2 at +0, zero tile, then the rest
      const uint32_t rWQ = rec + 2 * kT2 + (R::WQ - kT2);
      const uint32_t rAQ = rec + 2 * kT2 + (R::AQ - kT2);
      const uint32_t rKE = rec + 2 * kT2 + (R::KE - kT2);
      const uint32_t vt = sbase + L::VT + b * 64 * DV * 2;
      wait(mbar_rec0 + 8 * b, (ci >> 1) & 1);
      bar_sync(1, 160);
      // U/O buffer b was last used by chunk ci - 2: its output must have been read out
      if (ci >= 2) wait(mbar_orel0 + 8 * b, (uint32_t)(((ci - 2) >> 1) & 1));
      // [U ; Q+ S] = [T_beta | -W ; 0 | Q+] [V ; S]
      if (lane == 0) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tX(b), desc_kmajor(rec, 64, ks), desc_mnmajor(vt, 64, ks),
                   idesc_bf16(128, DV, false, true), ks > 0);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tX(b), desc_kmajor(rWQ, 128, ks), desc_mnmajor(sbase + L::SB, DK, ks),
                   idesc_bf16(128, DV, false, true), 1u);
        mma_commit(mbar_a);
      }
      __syncwarp();
      bar_sync(2, 160);
      // S += K_end^T U  (the state chain), then O += A_Q U (rows 64..127 of buffer b)
      if (lane == 0) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tS, desc_kmajor(rKE, DK, ks), desc_mnmajor(vt, 64, ks),
                   idesc_bf16(128, DV, false, true), 1u);
        mma_commit(mbar_s);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tX(b), desc_kmajor(rAQ - 64 * 128, 64, ks), desc_mnmajor(vt, 64, ks),
                   idesc_bf16(128, DV, false, true), 1u);
        mma_commit(mbar_free0 + 8 * b);  // chunk ci's output is ready; its buffers are free
      }
      __syncwarp();
    }
  } else {
    // ======================= TMEM <-> memory warps =======================
    // rows 64..127 of chunk pc's U/O buffer -> out (warps 2-3).  The values are
    // read from TMEM first and the buffer is released at once (orel, when
    // `release`); each warp then turns its 32 rows around through a small
    // shared staging area so that every store instruction writes four whole
    // 128-byte lines.
    auto store_out = [&](int pc, bool release) {
      const int lc = min(kC, rg.len - pc * kC);
      // 144-byte staging rows: consecutive rows start on different banks
      const uint32_t stage = sbase + L::OSTG + (warp - 2) * 32 * 144;
      uint32_t r[DV / 32][32];
#pragma unroll
      for (int q = 0; q < DV / 32; ++q) tmem_ld32_async(tX(pc & 1) + lane_base + 32 * q, r[q]);
      tmem_wait_ld();
      if (release) {
        fence_before_sync();
        mbar_arrive(mbar_orel0 + 8 * (pc & 1));
      }
      const int row0 = 32 * (warp - 2);  // this warp's first token row in the chunk
#pragma unroll
      for (int half = 0; half < DV / 64; ++half) {
        __syncwarp();  // the previous half has been read back
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float* f = reinterpret_cast<const float*>(r[2 * half + (u >> 2)]) + 8 * (u & 3);
          st_shared_v4(stage + lane * 144 + 16 * u, pack_bf16(a.scale * f[0], a.scale * f[1]),
                       pack_bf16(a.scale * f[2], a.scale * f[3]), pack_bf16(a.scale * f[4], a.scale * f[5]),
                       pack_bf16(a.scale * f[6], a.scale * f[7]));
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int rr = 4 * it + (lane >> 3), ch = lane & 7;
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(stage + rr * 144 + 16 * ch));
          const int t = row0 + rr;
          if (t < lc)
            *reinterpret_cast<uint4*>(og + ((int64_t)pc * kC + t) * a.out_st + 64 * half + 8 * ch) = w;
        }
      }
    };
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      const uint32_t rec = sbase + L::REC + b * L::kRecBuf;
      const uint32_t vt = sbase + L::VT + b * 64 * DV * 2;
      // (1) bf16 copy of the state entering this chunk (read once from TMEM, kept in registers)
      uint32_t r[DV / 32][32];
      if (ci > 0) wait(mbar_s, (uint32_t)((ci - 1) & 1));
      if (tid < DK) {
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) tmem_ld32_async(tS + lane_base + 32 * q, r[q]);
        tmem_wait_ld();
        if (ci > 0) {
#pragma unroll
          for (int q = 0; q < DV / 32; ++q)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(sbase + L::SB + sw128(tid, 32 * q + 8 * u, DK),
                           pack_bf16(__uint_as_float(r[q][8 * u]), __uint_as_float(r[q][8 * u + 1])),
                           pack_bf16(__uint_as_float(r[q][8 * u + 2]), __uint_as_float(r[q][8 * u + 3])),
                           pack_bf16(__uint_as_float(r[q][8 * u + 4]), __uint_as_float(r[q][8 * u + 5])),
                           pack_bf16(__uint_as_float(r[q][8 * u + 6]), __uint_as_float(r[q][8 * u + 7])));
        }
      }
      fence_async_smem();
      bar_arrive(1, 160);
      // (2) decay the TMEM state by e^{G_C} of this chunk (overlaps the first product)
      wait(mbar_rec0 + 8 * b, (ci >> 1) & 1);
      if (tid < DK) {
        const float pc = reinterpret_cast<const float*>(smem + (rec - sbase) + 2 * kT2 + (R::P - kT2))[tid];
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[q][i] = __float_as_uint(__uint_as_float(r[q][i]) * pc);
          tmem_st32_async(tS + lane_base + 32 * q, r[q]);
        }
        tmem_wait_st();
      }
      // (3) warps 0-1: U -> bf16 (MN-major [j][n]) into the consumed V buffer
      if (warp < 2) {
        wait(mbar_a, (uint32_t)(ci & 1));
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) tmem_ld32_async(tX(b) + lane_base + 32 * q, r[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < DV / 32; ++q)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(vt + sw128(tid, 32 * q + 8 * u, 64),
                         pack_bf16(__uint_as_float(r[q][8 * u]), __uint_as_float(r[q][8 * u + 1])),
                         pack_bf16(__uint_as_float(r[q][8 * u + 2]), __uint_as_float(r[q][8 * u + 3])),
                         pack_bf16(__uint_as_float(r[q][8 * u + 4]), __uint_as_float(r[q][8 * u + 5])),
                         pack_bf16(__uint_as_float(r[q][8 * u + 6]), __uint_as_float(r[q][8 * u + 7])));
        fence_async_smem();
      }
      fence_before_sync();
      bar_arrive(2, 160);
      // (4) warps 2-3: output of the previous chunk, then release its U/O buffer
      if (warp >= 2 && ci > 0) {
        wait(mbar_free0 + 8 * ((ci - 1) & 1), (uint32_t)(((ci - 1) >> 1) & 1));
        store_out(ci - 1, true);
      }
    }
    // last output and the final state
    if (nch > 0) {
      wait(mbar_s, (uint32_t)((nch - 1) & 1));
      if (warp >= 2) {
        wait(mbar_free0 + 8 * ((nch - 1) & 1), (uint32_t)(((nch - 1) >> 1) & 1));
        store_out(nch - 1, false);
      }
    }
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
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------
// chunk offsets of each sequence (varlen): off[n] = sum_{m < n} ceil(len_m / 64),
// capped at `total` so no record index can fall outside the workspace
__global__ void kda_chunk_offsets_kernel(PrefillArgs a, int total, int* off) {
  __shared__ int part[256];
  const int N = a.N;
  const int per = (N + 255) / 256;
  const int n0 = threadIdx.x * per;
  int s = 0;
  for (int i = 0; i < per; ++i) {
    const int n = n0 + i;
    if (n < N) s += (seq_range(a, n).len + kC - 1) / kC;
  }
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < 256; ++i) {
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
      off[n] = min(run, total);
      run += (seq_range(a, n).len + kC - 1) / kC;
    }
  }
}

int sm_count() {
  static int count = 0;
  if (!count) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
    if (count <= 0) count = 1;
  }
  return count;
}

template <int DK>
constexpr int rec_bytes() { return Rec<DK>::kBytes; }

int64_t split_total_chunks(const PrefillArgs& a) {
  const int64_t nck = ((int64_t)a.T + kC - 1) / kC;
  return a.cu_seqlens ? nck + a.N : nck * a.N;
}

template <int DK, int DV>
cudaError_t launch(const PrefillArgs& a, void* ws, cudaStream_t s) {
  const int64_t total = split_total_chunks(a);
  const int64_t off_bytes = a.cu_seqlens ? (((int64_t)(a.N + 1) * 4 + 1023) & ~int64_t(1023)) : 0;
  Split sp;
  sp.off = a.cu_seqlens ? static_cast<const int*>(ws) : nullptr;
  sp.rec = static_cast<unsigned char*>(ws) + off_bytes;
  sp.total = (int)total;
  sp.nck = (int)(((int64_t)a.T + kC - 1) / kC);
  cudaError_t e;
  if (a.cu_seqlens) {
    launch_begin(s);
    kda_chunk_offsets_kernel<<<1, 256, 0, s>>>(a, sp.total, static_cast<int*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  auto prep = kda_chunk_prep_kernel<DK>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, PrepSmem<DK>::kAlloc);
  if (e != cudaSuccess) return e;
  auto ser = kda_chunk_serial_kernel<DK, DV>;
  e = cudaFuncSetAttribute(ser, cudaFuncAttributeMaxDynamicSharedMemorySize, SerialSmem<DK, DV>::kAlloc);
  if (e != cudaSuccess) return e;
  const int64_t items = total * a.H;
  const int grid = (int)(items < 2 * sm_count() ? items : 2 * sm_count());
  if (grid > 0) {
    launch_begin(s);
    prep<<<grid, kThreads, PrepSmem<DK>::kAlloc, s>>>(a, sp);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  launch_begin(s);
  ser<<<dim3((unsigned)(a.N * a.H)), kSerialThreads, SerialSmem<DK, DV>::kAlloc, s>>>(a, sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

}  // namespace

size_t chunk_prefill_workspace_bytes(const PrefillArgs& a) {
  const int64_t total = split_total_chunks(a);
  const int64_t off_bytes = a.cu_seqlens ? (((int64_t)(a.N + 1) * 4 + 1023) & ~int64_t(1023)) : 0;
  const int64_t rb = a.dk == 128 ? rec_bytes<128>() : rec_bytes<64>();
  return (size_t)(off_bytes + total * a.H * rb);
}

cudaError_t launch_chunk_prefill_tc(const PrefillArgs& a, void* workspace, cudaStream_t s) {
  if (!a.bf16) return cudaErrorInvalidValue;
  if (a.dk == 128 && a.dv == 128) return launch<128, 128>(a, workspace, s);
  if (a.dk == 128 && a.dv == 64) return launch<128, 64>(a, workspace, s);
  if (a.dk == 64 && a.dv == 128) return launch<64, 128>(a, workspace, s);
  if (a.dk == 64 && a.dv == 64) return launch<64, 64>(a, workspace, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
