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
//     K e^{G_C - G} -- plus e^{G_C} to a workspace.  Tiles that come out of
//     TMEM or the solve are staged in shared memory and leave by bulk copy.
//   * kda_chunk_serial_kernel: one CTA per (sequence, head, slice of 32, 64 or
//     all d_v value columns -- the state's columns evolve independently) keeps
//     its fp32 state columns in TMEM and walks the chunks in order, with warp
//     roles: a producer warp
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
//     The column operand exists in 4 versions (16, 32, 48, 64 rows), stacked as
//     one 160-row operand; one product covers all 128 rows [K; Q] against all
//     versions, and row block I keeps only version I's columns.
//   * K+ = K e^{G}, Q+ = Q e^{G}, K e^{G_C - G} are all <= 1.
//
// Several M = 128 products only use 64 meaningful A rows: their descriptor
// window extends over a neighbouring tile, and the corresponding accumulator
// rows are never read (or are overwritten before they are read).
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kThreads = 256;  // prep kernel
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }

// One chunk record (per chunk and head), byte offsets.  Tiles are stored exactly
// as they sit in shared memory, so one bulk copy moves the whole record.
template <int DK>
struct Rec {
  static constexpr int T2 = 0;                      // T Diag(beta): 64 x 64, K-major
  static constexpr int WQ = T2 + 64 * 64 * 2;       // [-W ; Q+]: 128 x DK, K-major
  static constexpr int AQ = WQ + 128 * DK * 2;      // A_Q: 64 x 64, K-major
  static constexpr int KE = AQ + 64 * 64 * 2;       // K e^{G_C - G}: 64 x DK, MN-major (A of S += K_end^T U)
  static constexpr int P = KE + 64 * DK * 2;        // e^{G_C}: DK fp32
  static constexpr int kBytes = align1k(P + DK * 4);
};

// Gram column versions: version I has 16 (I + 1) rows, stacked in order.
__host__ __device__ constexpr int yoff_rows(int I) { return 8 * I * (I + 1); }  // rows before version I

// Decay-factor table of the prep kernel: entry (a, b), a < b <= 4, holds
// 2^(bnd[b] - bnd[a]) per channel, bnd[x] being the cumulative log2-decay before
// sub-block x (bnd[4]: at the chunk end).
__host__ __device__ constexpr int ft_index(int a, int b) { return a * (9 - a) / 2 + (b - a - 1); }

template <int DK>
struct PrepSmem {
  static constexpr int kParts = kThreads / (DK / 8);   // token parts of the build
  // region shared by the Gram operands and, after the Gram product, the solve
  static constexpr int X = 0;                          // 128 rows [K; Q] x DK, K-major
  static constexpr int Y = X + 128 * DK * 2;           // versions 0..3 stacked: one 160-row K-major tile
  static constexpr int kGram = Y + 160 * DK * 2;
  static constexpr int CARRY = 0;                      // scan partials [part][DK] fp32 (before X is built)
  static_assert(kParts * DK * 4 <= 128 * DK * 2, "scan partials fit below Y");
  static constexpr int kLd = 68;  // fp32 row stride of L
  static constexpr int kTd = 72;  // fp32 row stride of T
  static constexpr int kRd = 40;  // fp32 row stride of the product scratch
  static constexpr int SL = 0;
  static constexpr int ST = SL + 64 * kLd * 4;
  static constexpr int SR = ST + 64 * kTd * 4;         // 32 x kRd
  static constexpr int T2 = align1k(SR + 32 * kRd * 4);  // 64 x 64 bf16 (+ an 8K window)
  static constexpr int AQS = T2 + 64 * 64 * 2;  // A_Q staging: the window below T2, whose
                                                // product rows are never read
  static constexpr int kSolve = T2 + 2 * 64 * 64 * 2;
  static constexpr int kG = kGram > kSolve ? kGram : kSolve;
  static constexpr int KP = align1k(kG);  // K+ : [64 tokens][DK], MN-major
  static constexpr int BETA = KP + 64 * DK * 2;
  static constexpr int BND = BETA + 64 * 4;   // 5 x DK fp32 (log2 units)
  static constexpr int FT = BND + 5 * DK * 4; // 10 x DK fp32 decay factors
  static constexpr int MBAR = FT + 10 * DK * 4;  // MMA completion, then the exit drain
  static constexpr int TSLOT = MBAR + 16;
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
  // MN-major tiles keep 128-byte rows (the swizzle atom) when DV = 32: the 32
  // columns occupy half of each row's 16-byte chunks, at their swizzled places
  static constexpr int kPitch = DV < 64 ? 64 : DV;       // stored columns of a value tile
  static constexpr int REC = 0;                          // two record buffers
  static constexpr int VT = REC + 2 * kRecBuf;           // two V chunks [64][DV] MN-major (U reuses)
  static constexpr int SB = VT + 2 * 64 * kPitch * 2;    // bf16 S, [DK][DV] MN-major
  static constexpr int OSTG = SB + DK * kPitch * 2;      // output staging: 2 warps x 32 rows x 144 B
  static constexpr int MBAR = OSTG + 2 * 32 * 144;       // mma_a, mma_s, rec0/1, free0/1, orel0/1, done
  static constexpr int TSLOT = MBAR + 72;
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

// Segment split of long sequences.  A sequence of more than kFirstSeg chunks is
// cut into a first segment of kFirstSeg chunks and tail segments of kTailSeg
// chunks, counted from its start (so the cut depends on the sequence alone).
// Segment 0 runs from the initial state.  Each tail segment s first runs from
// zero on the augmented state [S~ | M], which starts as [0 | I] with values
// [V | 0]: M then equals the product of the chunk transitions
// Diag(e^{G_C}) - K_end^T W over the segment and S~ the segment's result from a
// zero state.  The states entering the tail segments follow in order,
// S_in(s + 1) = M_s S_in(s) + S~_s, and a second pass reruns the tail segments
// from them, writing their outputs.  Every chunk past the first segment is run
// twice, however the tail is cut; short tail segments give both passes more,
// shorter units to spread over the SMs.
constexpr int kFirstSeg = 1152;
constexpr int kTailSeg = 128;
static_assert(kTailSeg <= kFirstSeg, "the tail-unit bound of the workspace plan");

struct Seg {
  float* tr;        // [tail unit][H][DK][dv + DK] fp32: (S~ | M) of each tail segment
  float* sin;       // [tail unit][H][DK][dv] fp32: state entering each tail segment
  const int* soff;  // tail segments before sequence n ([N + 1]); null for fixed length
  int ntail;        // tail units allocated
  int tps;          // tail segments per sequence (fixed length)
};

__host__ __device__ __forceinline__ int num_segments(int nc) {
  return nc > kFirstSeg ? 1 + (nc - kFirstSeg + kTailSeg - 1) / kTailSeg : 1;
}
__device__ __forceinline__ int tail_first(const Seg& sg, int n) { return sg.soff ? __ldg(sg.soff + n) : n * sg.tps; }
__device__ __forceinline__ int tail_count(const Seg& sg, int N) {
  return sg.soff ? min(__ldg(sg.soff + N), sg.ntail) : N * sg.tps;
}
// sequence of tail unit u (u < tail_count)
__device__ __forceinline__ int tail_seq(const Seg& sg, int N, int u) {
  if (!sg.soff) return u / sg.tps;
  int lo = 0, hi = N - 1;  // largest n with soff[n] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(sg.soff + mid) <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
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

// 1/x on the special-function unit (relative error ~2^-23; 1/inf = 0).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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
// C (16 x 8 tile) = sum over k in [k0, k1) of A[row][k] B[k][col] on one warp
// (m16n8k8, tf32 inputs, fp32 accumulation).  A and B are fp32 in shared memory,
// A's tile starting at `A` with row stride lda, B's at `B` with row stride ldb.
__device__ __forceinline__ void warp_tile_tf32(float (&acc)[4], const float* A, int lda, const float* B,
                                               int ldb, int k0, int k1, int lane) {
  const int g = lane >> 2, t = lane & 3;
  for (int k = k0; k < k1; k += 8) {
    const uint32_t af[4] = {to_tf32(A[g * lda + k + t]), to_tf32(A[(g + 8) * lda + k + t]),
                            to_tf32(A[g * lda + k + t + 4]), to_tf32(A[(g + 8) * lda + k + t + 4])};
    const uint32_t bf[2] = {to_tf32(B[(k + t) * ldb + g]), to_tf32(B[(k + t + 4) * ldb + g])};
    mma_tf32(acc, af, bf);
  }
}

// Store a 16 x 8 accumulator tile (times `sign`) at C (row stride ldc).
__device__ __forceinline__ void warp_tile_store(const float (&acc)[4], float* C, int ldc, float sign, int lane) {
  const int g = lane >> 2, t = lane & 3;
  C[g * ldc + 2 * t] = sign * acc[0];
  C[g * ldc + 2 * t + 1] = sign * acc[1];
  C[(g + 8) * ldc + 2 * t] = sign * acc[2];
  C[(g + 8) * ldc + 2 * t + 1] = sign * acc[3];
}

// ---------------------------------------------------------------------------
// prep: one chunk of one head per iteration; persistent CTAs of 8 warps, two per SM
template <int DK, bool GATE>
__global__ void __launch_bounds__(kThreads, 2) kda_chunk_prep_kernel(PrefillArgs a, Split sp) {
  using L = PrepSmem<DK>;
  using R = Rec<DK>;
  constexpr int OCT = DK / 8;            // channel octets
  constexpr int NPART = kThreads / OCT;  // token parts in the build
  constexpr int TPP = 64 / NPART;        // tokens per part (4 or 2)
  constexpr int PPB = 16 / TPP;          // parts per 16-token sub-block
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
  float* sFt = reinterpret_cast<float*>(smem + L::FT);
  float* sCarry = reinterpret_cast<float*>(smem + L::CARRY);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + L::FLAG);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter

  if (tid == 0) {
    mbar_init(sbase + L::MBAR, 1);
    mbar_init(sbase + L::MBAR + 8, 1);
    fence_mbar_init();
    *sFlag = 0;
  }
  if (warp == 0) tmem_alloc(sbase + L::TSLOT, L::kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);
  Ctx ctx{sbase + L::MBAR, 0u, sFlag, a.err};
  // the serial kernel may be launched now (it waits for this grid before it reads
  // any record), so its CTAs set up on SMs this grid leaves early
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int oct = tid % OCT;
  const int part = tid / OCT;
  const int blk = part / PPB;  // this part's 16-token sub-block
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
  float4 rg[TPP][2];  // log-decay (fp32), or
  uint4 rz[TPP];      // decay logits (bf16) with the gate
  float rbeta = 0.f;
  float gsc = 0.f;    // gate scale of the current head
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
    if constexpr (GATE) {
      const __nv_bfloat16* zb = static_cast<const __nv_bfloat16*>(a.g.ptr) + it.brow * a.g.sb + it.h * a.g.sh;
#pragma unroll
      for (int i = 0; i < TPP; ++i) {
        const int t = part * TPP + i;
        const bool ok = it.valid && t < it.lc;
        const int64_t row = it.row0 + t;
        rz[i] = ok ? __ldg(reinterpret_cast<const uint4*>(zb + row * a.g.st) + oct) : make_uint4(0, 0, 0, 0);
      }
    } else {
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
    }
    const float* bb = a.beta + it.brow * a.beta_sb + it.h * a.beta_sh;
    rbeta = (it.valid && tid < it.lc) ? __ldg(bb + (it.row0 + tid) * a.beta_st) : 0.f;
    if constexpr (GATE) gsc = it.valid ? __ldg(a.gate_scale + it.h) : 0.f;
  };
  auto pack8 = [](const float* x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
  };
  auto st8 = [&](uint32_t addr, const float* x) {
    const uint4 u = pack8(x);
    st_shared_v4(addr, u.x, u.y, u.z, u.w);
  };
  // 8 consecutive fp32 of shared memory (16-byte aligned)
  auto ld8 = [](const float* p, float* x) {
    const float4 u = reinterpret_cast<const float4*>(p)[0], v = reinterpret_cast<const float4*>(p)[1];
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
  };
  auto bf16x8 = [](const uint4& w, float* x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (e & 1) ? bf_hi(u[e >> 1]) : bf_lo(u[e >> 1]);
  };

  Item cur = item(blockIdx.x);
  load_kq(cur);
  load_g(cur);

  for (int w = blockIdx.x; w < nitems; w += gridDim.x) {
    Item nxt;  // placed while the Gram product runs, where its loads are hidden
    if (cur.valid) {
      unsigned char* rec = sp.rec + cur.rec * R::kBytes;
      const int col = 8 * oct;

      // ================= scan: G (log2 units), 8 channels x TPP tokens per thread =================
      float G[TPP][8];
      {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < TPP; ++i) {
          float gv[8];
          if constexpr (GATE) {
            // g = -5 sigmoid(A_h z) = -5 / (1 + 2^(-A_h z log2 e)); an infinite
            // power gives a zero reciprocal, so g -> -0 for very negative A_h z.
            // Tokens past the chunk's end (padding) keep g = 0.
            float zf[8];
            bf16x8(rz[i], zf);
            const bool real = part * TPP + i < cur.lc;
#pragma unroll
            for (int e = 0; e < 8; ++e) gv[e] = real ? -5.f * rcp_approx(1.f + ex2(-kLog2e * gsc * zf[e])) : 0.f;
          } else {
            gv[0] = rg[i][0].x; gv[1] = rg[i][0].y; gv[2] = rg[i][0].z; gv[3] = rg[i][0].w;
            gv[4] = rg[i][1].x; gv[5] = rg[i][1].y; gv[6] = rg[i][1].z; gv[7] = rg[i][1].w;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            acc[e] = fmaf(gv[e], kLog2e, acc[e]);
            G[i][e] = acc[e];
          }
        }
        float4* cw = reinterpret_cast<float4*>(sCarry + part * DK + col);
        cw[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        cw[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (tid < 64) sBeta[tid] = rbeta;
      }
      __syncthreads();
      // one thread per channel: exclusive prefix over the parts, the sub-block
      // boundaries, e^{G_C} (record) and the decay-factor table
      if (tid < DK) {
        const int c = tid;
        float v[NPART];
#pragma unroll
        for (int p = 0; p < NPART; ++p) v[p] = sCarry[p * DK + c];
        float run = 0.f, bnd[5];
#pragma unroll
        for (int p = 0; p < NPART; ++p) {
          if (p % PPB == 0) bnd[p / PPB] = run;
          sCarry[p * DK + c] = run;
          run += v[p];
        }
        bnd[4] = run;
#pragma unroll
        for (int x = 0; x < 5; ++x) sBnd[x * DK + c] = bnd[x];
        reinterpret_cast<float*>(rec + R::P)[c] = exp2f(run);
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = x + 1; y <= 4; ++y) sFt[ft_index(x, y) * DK + c] = ex2(bnd[y] - bnd[x]);
      }
      __syncthreads();
      {
        // G relative to the start of this thread's sub-block
        float off[8], b0[8];
        ld8(sCarry + part * DK + col, off);
        ld8(sBnd + blk * DK + col, b0);
#pragma unroll
        for (int i = 0; i < TPP; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) G[i][e] += off[e] - b0[e];
      }
      // the previous item's bulk copies must have read their staging tiles (which
      // the build overwrites); the scan partials share memory with X
      if (tid == 0) bulk_wait_read0();
      __syncthreads();

      // ================= build: the Gram operands =================
      // Rows use the reference G at the start of sub-block blk: X = k e^{G - bnd[blk]}
      // (and q).  Column version J >= blk uses the reference at the start of
      // sub-block J: k e^{bnd[J] - G}.  These feed the Gram product; Q+ = q e^{G} goes to
      // the record on the way, and the tiles not needed until later (K+, K_end) are
      // formed while the product runs.
      float fbl[8];  // 2^{bnd[blk]}: from the sub-block reference to the chunk start
      if (blk > 0) {
        ld8(sFt + ft_index(0, blk) * DK + col, fbl);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) fbl[e] = 1.f;
      }
      {
        // q rows: Gram rows 64.., and Q+ (record)
#pragma unroll
        for (int i = 0; i < TPP; ++i) {
          const int t = part * TPP + i;
          float x[8];
          bf16x8(rq[i], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= ex2(G[i][e]);
          st8(sbase + L::X + sw128(64 + t, col, 128), x);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= fbl[e];
          *reinterpret_cast<uint4*>(rec + R::WQ + sw128(64 + t, col, 128)) = pack8(x);
        }
        // k rows; y = k e^{bnd[blk] - G} for the column versions
        float y[TPP][8];
#pragma unroll
        for (int i = 0; i < TPP; ++i) {
          const int t = part * TPP + i;
          float kv[8], x[8];
          bf16x8(rk[i], kv);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = kv[e] * ex2(G[i][e]);
          st8(sbase + L::X + sw128(t, col, 128), x);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[i][e] = kv[e] * ex2(-G[i][e]);
        }
        // column version J >= blk: y 2^{bnd[J] - bnd[blk]}
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          if (J < blk) continue;
          float f[8];
          if (J > blk) {
            ld8(sFt + ft_index(blk, J) * DK + col, f);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 1.f;
          }
#pragma unroll
          for (int i = 0; i < TPP; ++i) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[i][e] * f[e];
            st8(sbase + L::Y + sw128(yoff_rows(J) + part * TPP + i, col, 160), x);
          }
        }
      }
      fence_async_smem();
      fence_before_sync();
      __syncthreads();

      // ================= Gram: all 128 rows [K; Q] against the four column versions =================
      // (one N = 160 product; row block I later reads only version I's columns)
      if (tid == 0) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tmem, desc_kmajor(sbase + L::X, 128, ks), desc_kmajor(sbase + L::Y, 160, ks),
                   idesc_bf16(128, 160, false, false), ks > 0);
        mma_commit(ctx.mbar);
      }
      // ---- while the product runs: K_end = k e^{G_C - G} (record, token rows) and
      // K+ = k e^{G} (shared memory, for W), from the same registers ----
      {
        float fend[8];
        ld8(sFt + ft_index(blk, 4) * DK + col, fend);
#pragma unroll
        for (int i = 0; i < TPP; ++i) {
          const int t = part * TPP + i;
          float x[8], kv[8], y[8];
          bf16x8(rk[i], kv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = kv[e] * ex2(G[i][e]) * fbl[e];
            y[e] = kv[e] * ex2(-G[i][e]) * fend[e];
          }
          st8(sbase + L::KP + sw128(t, col, 64), x);
          *reinterpret_cast<uint4*>(rec + R::KE + sw128(t, col, 64)) = pack8(y);
        }
        fence_async_smem();  // K+ is read by the W product, several barriers later
      }
      // the k/q registers are free: start loading the next item while the MMAs run
      nxt = item(w + gridDim.x);
      load_kq(nxt);
      wait_mma(ctx);

      // ---- Gram epilogue: TMEM lane r < 64 -> row r of L (fp32); lane 64 + r -> row r of A_Q ----
      // Warp w reads lane quarter w & 3 and the column version b of one of its two
      // row blocks (warps 4-7 take the second).
      {
        const int quarter = warp & 3;
        const int i = (32 * quarter + lane) & 63;
        const int myblk = i >> 4;
        const int b = (quarter & 1) * 2 + (warp >> 2);
        for (int pc = 0; pc <= b; ++pc) {  // 16-column pieces of version b
          float v[16];
          tmem_ld16(tmem + lane_base + yoff_rows(b) + 16 * pc, v);
          if (myblk == b) {
            const int j0 = 16 * pc;
            if (quarter < 2) {
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
                st8(sbase + L::AQS + sw128(i, j0 + 8 * u, 64), x);
              }
            }
          }
        }
        if (quarter >= 2 && myblk == b) {  // A_Q columns past this row's sub-block are zero
          for (int j0 = 16 * (myblk + 1); j0 < 64; j0 += 8)
            st_shared_v4(sbase + L::AQS + sw128(i, j0, 64), 0u, 0u, 0u, 0u);
        }
        fence_async_smem();
      }
      __syncthreads();
      if (tid == 0) bulk_s2g(rec + R::AQ, sbase + L::AQS, 64 * 64 * 2);

      // ================= T = (I + L)^-1 (fp32) =================
      if (tid < 64) {  // diagonal 16 x 16 blocks by substitution, one column per thread
        const int I = tid >> 4, cc = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float s0 = (r == cc) ? 1.f : 0.f, s1 = 0.f;
          const float4* lr = reinterpret_cast<const float4*>(sL + (16 * I + r) * L::kLd + 16 * I);
#pragma unroll
          for (int m4 = 0; m4 < r; m4 += 4) {  // L[r][m] for m < r (entries at m >= r are zero)
            const float4 l = lr[m4 >> 2];
            s0 -= l.x * x[m4];
            if (m4 + 1 < r) s1 -= l.y * x[m4 + 1];
            if (m4 + 2 < r) s0 -= l.z * x[m4 + 2];
            if (m4 + 3 < r) s1 -= l.w * x[m4 + 3];
          }
          x[r] = (r > cc) ? s0 + s1 : ((r == cc) ? 1.f : 0.f);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(16 * I + r) * L::kTd + 16 * I + cc] = x[r];
      }
      __syncthreads();
      // Off-diagonal blocks by doubling, on the warp-level tensor cores (tf32):
      //   16 -> 32:  T[2p+1, 2p] = -D_{2p+1} (L[2p+1, 2p] D_{2p})        (p = 0, 1)
      //   32 -> 64:  T[B, A] = -T_BB (L_BA T_AA),  A = rows 0-31, B = rows 32-63
      // Blocks of T above the diagonal are never read (they hold stale values).
      if (warp < 4) {  // R_p = L[2p+1, 2p] D_{2p}: 16 x 16, two column tiles each
        const int p = warp >> 1, nt = warp & 1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_tile_tf32(acc, sL + (32 * p + 16) * L::kLd + 32 * p, L::kLd, sT + (32 * p) * L::kTd + 32 * p + 8 * nt,
                       L::kTd, 0, 16, lane);
        warp_tile_store(acc, sR + (16 * p) * L::kRd + 8 * nt, L::kRd, 1.f, lane);
      }
      __syncthreads();
      if (warp < 4) {  // T[2p+1, 2p] = -D_{2p+1} R_p
        const int p = warp >> 1, nt = warp & 1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_tile_tf32(acc, sT + (32 * p + 16) * L::kTd + 32 * p + 16, L::kTd, sR + (16 * p) * L::kRd + 8 * nt,
                       L::kRd, 0, 16, lane);
        warp_tile_store(acc, sT + (32 * p + 16) * L::kTd + 32 * p + 8 * nt, L::kTd, -1.f, lane);
      }
      __syncthreads();
      {  // X = L_BA T_AA (32 x 32): warp -> row tile mt, column tile nt; T_AA is block lower triangular
        const int mt = warp >> 2, nt = warp & 3;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_tile_tf32(acc, sL + (32 + 16 * mt) * L::kLd, L::kLd, sT + 8 * nt, L::kTd, nt >= 2 ? 16 : 0, 32, lane);
        warp_tile_store(acc, sR + (16 * mt) * L::kRd + 8 * nt, L::kRd, 1.f, lane);
      }
      __syncthreads();
      {  // T_BA = -T_BB X: T_BB is block lower triangular
        const int mt = warp >> 2, nt = warp & 3;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        warp_tile_tf32(acc, sT + (32 + 16 * mt) * L::kTd + 32, L::kTd, sR + 8 * nt, L::kRd, 0, 16 * (mt + 1), lane);
        warp_tile_store(acc, sT + (32 + 16 * mt) * L::kTd + 8 * nt, L::kTd, -1.f, lane);
      }
      __syncthreads();
      // the next item's decay rows: issued here, a few phases before its scan reads
      // them (issued later they arrive too late; earlier, the registers they hold
      // push the inverse's live values into local memory)
      load_g(nxt);
      // T_beta = T Diag(beta) -> bf16 K-major [i][j] in shared memory (and the record, by bulk copy)
      {
        const int i = tid >> 2, j0 = 16 * (tid & 3);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float tv[8], bv[8], x[8];
          ld8(sT + i * L::kTd + j0 + 8 * u, tv);
          ld8(sBeta + j0 + 8 * u, bv);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = (j0 + 8 * u + e <= i) ? tv[e] * bv[e] : 0.f;
          st8(sbase + L::T2 + sw128(i, j0 + 8 * u, 64), x);
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
        bulk_s2g(rec + R::T2, sbase + L::T2, 64 * 64 * 2);
      }
      wait_mma(ctx);
      // ---- -W (bf16, rows 0..63 of the [-W ; Q+] tile) staged over K+ (free once W is
      // done), then one bulk copy per 64-column panel.  Lane quarters 0-1; warps 4-5
      // take the upper columns. ----
      if ((warp & 3) < 2) {
        const int r = 32 * (warp & 3) + lane;
        const int c_lo = (warp >> 2) * (DK / 2);
#pragma unroll
        for (int c0 = c_lo; c0 < c_lo + DK / 2; c0 += 32) {
          float v[32];
          tmem_ld32(tmem + lane_base + c0, v);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = -v[8 * u + e];
            st8(sbase + L::KP + sw128(r, c0 + 8 * u, 64), x);
          }
        }
        fence_async_smem();
      }
      fence_before_sync();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int pn = 0; pn < DK / 64; ++pn)  // panel pn: 64 rows x 128 B, at pn * 128 rows in the record
          bulk_s2g(rec + R::WQ + pn * 128 * 128, sbase + L::KP + pn * 64 * 128, 64 * 128);
        bulk_commit();
      }
      if (*sFlag) break;
    } else {
      nxt = item(w + gridDim.x);
      load_kq(nxt);
      load_g(nxt);
    }
    cur = nxt;
  }
  if (tid == 0) {
    bulk_wait0();  // this CTA's record writes are complete
    // every product this thread issued has completed before TMEM is freed (after a
    // timed-out wait one may still be running; otherwise this returns at once)
    mma_commit(sbase + L::MBAR + 8);
    if (!mbar_wait(sbase + L::MBAR + 8, 0)) atomicOr(a.err, kErrTimeout);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------
// serial: one (sequence, head, value-column slice) per CTA, fp32 state in TMEM.
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

// What one serial CTA computes: DV columns of one (sequence, head) state over the
// chunk range [c0, c1) of the sequence.
struct Unit {
  int n, h;
  int c0, c1;
  int kind;            // 0: value columns (outputs); 1: tail pass 1, S~ columns; 2: tail pass 1, M columns
  int col;             // first value column (kinds 0 and 1)
  int m0;              // first M column (kind 2)
  const float* init;   // initial state rows, row stride init_ld; null = zero (kinds 0, 1)
  int64_t init_ld;
  float* fin;          // where the final state rows go (row stride fin_ld), or null
  int64_t fin_ld;
  int fin_cols;        // columns of fin to write
};

// CTA -> unit.  pass 0: first the units of every sequence's first segment (value
// column slices), then, per tail unit and head, slices of the DV + DK augmented
// columns; pass 1: per tail unit and head, value column slices.  Returns false for
// CTAs past the tail units in use.
template <int DK, int DV>
__device__ __forceinline__ bool serial_unit(const PrefillArgs& a, const Split& sp, const Seg& sg, int pass, int bid,
                                            Unit& u) {
  const int nsl = a.dv / DV;  // value column slices per (sequence, head)
  const int nfirst = a.N * a.H * nsl;
  if (pass == 0 && bid < nfirst) {
    const int sl = bid % nsl, nh = bid / nsl;
    u.n = nh / a.H;
    u.h = nh - u.n * a.H;
    const Range rg = seq_range(a, u.n);
    const int nc = min(num_chunks(sp, u.n), (rg.len + kC - 1) / kC);
    u.c0 = 0;
    u.c1 = min(nc, kFirstSeg);
    u.kind = 0;
    u.col = sl * DV;
    u.m0 = 0;
    u.init = a.s0 ? a.s0 + u.n * a.s0_sn + u.h * a.s0_sh + u.col : nullptr;
    u.init_ld = a.dv;
    u.fin_ld = a.dv;
    u.fin_cols = DV;
    if (num_segments(nc) == 1) {
      u.fin = a.sT ? a.sT + u.n * a.sT_sn + u.h * a.sT_sh + u.col : nullptr;
    } else {
      const int t = tail_first(sg, u.n);
      u.fin = t < tail_count(sg, a.N) ? sg.sin + ((int64_t)t * a.H + u.h) * DK * a.dv + u.col : nullptr;
    }
    return true;
  }
  const int t = pass == 0 ? bid - nfirst : bid;
  const int nx = pass == 0 ? (a.dv + DK + DV - 1) / DV : nsl;  // column slices of a tail unit
  const int xs = t % nx, uh = t / nx;
  u.h = uh % a.H;
  const int ut = uh / a.H;
  if (ut >= tail_count(sg, a.N)) return false;
  u.n = tail_seq(sg, a.N, ut);
  const Range rg = seq_range(a, u.n);
  const int nc = min(num_chunks(sp, u.n), (rg.len + kC - 1) / kC);
  const int sgi = ut - tail_first(sg, u.n) + 1;  // segment index (>= 1)
  u.c0 = kFirstSeg + (sgi - 1) * kTailSeg;
  u.c1 = min(nc, u.c0 + kTailSeg);
  u.m0 = 0;
  if (pass == 0) {
    const int x0 = xs * DV;
    u.fin = sg.tr + ((int64_t)ut * a.H + u.h) * DK * (a.dv + DK) + x0;
    u.fin_ld = a.dv + DK;
    u.fin_cols = min(DV, a.dv + DK - x0);
    u.init = nullptr;
    u.init_ld = 0;
    if (x0 < a.dv) {
      u.kind = 1;
      u.col = x0;
    } else {
      u.kind = 2;
      u.col = 0;
      u.m0 = x0 - a.dv;
    }
  } else {
    u.kind = 0;
    u.col = xs * DV;
    u.init = sg.sin + ((int64_t)ut * a.H + u.h) * DK * a.dv + u.col;
    u.init_ld = a.dv;
    u.fin = (sgi == num_segments(nc) - 1 && a.sT) ? a.sT + u.n * a.sT_sn + u.h * a.sT_sh + u.col : nullptr;
    u.fin_ld = a.dv;
    u.fin_cols = DV;
  }
  return true;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kSerialThreads, 1)
    kda_chunk_serial_kernel(PrefillArgs a, Split sp, Seg sg, int pass) {
  Unit un;
  if (!serial_unit<DK, DV>(a, sp, sg, pass, blockIdx.x, un)) return;  // CTA-uniform
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
  const uint32_t mbar_done = mbar_a + 64;   // exit drain: every product issued has completed
  constexpr int kT2 = 64 * 64 * 2;  // T2 tile bytes; the rest of a record lands after the zero tile
  // Bounded waits.  With a.test_stall (tests of the timeout path only) the producer
  // issues no copies and every wait gives up after about 0.1 ms.
  const long long wait_limit = a.test_stall ? 200000ll : 4000000000ll;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  // The state's columns evolve independently, so a CTA owns DV columns of one
  // (sequence, head) state over a range of its chunks.
  const int n = un.n, h = un.h;
  const Range rg = seq_range(a, n);
  const int c0 = un.c0;         // chunk ci of this CTA is chunk c0 + ci of the sequence
  const int nch = un.c1 - un.c0;
  const bool vzero = un.kind == 2;  // M columns: no values
  const bool outs = un.kind == 0;
  // record of the sequence's chunk c: rec0 + c * H
  const int64_t rec0 = (int64_t)first_chunk(sp, n) * a.H + h;

  const __nv_bfloat16* vg =
      static_cast<const __nv_bfloat16*>(a.v.ptr) + rg.brow * a.v.sb + rg.tok0 * a.v.st + h * a.v.sh + un.col;
  __nv_bfloat16* og =
      static_cast<__nv_bfloat16*>(a.out) + rg.brow * a.out_sb + rg.tok0 * a.out_st + h * a.out_sh + un.col;

  if (tid == 0) {
    mbar_init(mbar_a, 1);
    mbar_init(mbar_s, 1);
    mbar_init(mbar_rec0, 33);  // producer lane 0's expect_tx arrival + 32 cp.async arrivals
    mbar_init(mbar_rec0 + 8, 33);
    mbar_init(mbar_free0, 1);
    mbar_init(mbar_free0 + 8, 1);
    mbar_init(mbar_orel0, 64);  // every thread of warps 2-3
    mbar_init(mbar_orel0 + 8, 64);
    mbar_init(mbar_done, 1);
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
  // Bounded wait.  After any timeout the abort flag is up: every later wait returns
  // at once, and no role issues further asynchronous work (products, copies), but
  // every role still walks its loop through the named barriers, so all finish.
  auto wait = [&](uint32_t mbar, uint32_t parity) {
    if (!*sFlag && !mbar_wait(mbar, parity, wait_limit)) {
      atomicOr(a.err, kErrTimeout);
      *sFlag = 1;
    }
    fence_after_sync();
  };

  if (tid < DK) {  // lane c holds state row c: TMEM <- initial state, shared <- its bf16 copy
    const float* s0 = un.init ? un.init + (int64_t)tid * un.init_ld : nullptr;
#pragma unroll
    for (int cb = 0; cb < DV; cb += 32) {
      float v[32];
      if (un.kind == 2) {  // identity columns m0 .. m0 + DV - 1 of M (zero past DK)
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = (tid == un.m0 + cb + i) ? 1.f : 0.f;
      } else {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + cb + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = x.x;
          v[i + 1] = x.y;
          v[i + 2] = x.z;
          v[i + 3] = x.w;
        }
      }
      tmem_st32(tS + lane_base + cb, v);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4(sbase + L::SB + sw128(tid, cb + 8 * u, DK), pack_bf16(v[8 * u], v[8 * u + 1]),
                     pack_bf16(v[8 * u + 2], v[8 * u + 3]), pack_bf16(v[8 * u + 4], v[8 * u + 5]),
                     pack_bf16(v[8 * u + 6], v[8 * u + 7]));
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();

  if (warp == 5) {
    // ======================= producer warp =======================
    // the records come from the previous grid (launched with programmatic
    // serialization): wait until it has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int last[2] = {-1, -1};  // last chunk whose copies were issued into each buffer
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      if (ci >= 2) wait(mbar_free0 + 8 * b, (uint32_t)(((ci - 2) >> 1) & 1));  // chunk ci - 2 is done
      // one decision for the whole warp: after an abort nothing more is issued
      if (__shfl_sync(0xffffffffu, (a.test_stall || *sFlag) ? 1 : 0, 0)) continue;
      last[b] = ci;
      const uint32_t dst = sbase + L::REC + b * L::kRecBuf;
      const uint32_t mb = mbar_rec0 + 8 * b;
      if (lane == 0) {
        const unsigned char* src = sp.rec + (rec0 + (int64_t)(c0 + ci) * a.H) * R::kBytes;
        if (outs) {
          mbar_arrive_expect_tx(mb, R::kBytes);
          bulk_g2s(dst, src, kT2, mb);
          bulk_g2s(dst + 2 * kT2, src + kT2, R::kBytes - kT2, mb);
        } else {
          // no outputs: A_Q and the Q+ rows of [-W ; Q+] are not needed, nor T_beta
          // without values.  -W is rows 0-63 of each 128-row panel of that tile.
          constexpr uint32_t kHalfPanel = 64 * 128, kPanel = 2 * kHalfPanel;
          constexpr uint32_t kTail = R::kBytes - R::KE;  // K_end and e^{G_C}
          const uint32_t rw = dst + 2 * kT2 + (R::WQ - kT2);
          mbar_arrive_expect_tx(mb, (vzero ? 0u : (uint32_t)kT2) + 2 * kHalfPanel + kTail);
          if (!vzero) bulk_g2s(dst, src, kT2, mb);
          bulk_g2s(rw, src + R::WQ, kHalfPanel, mb);
          bulk_g2s(rw + kPanel, src + R::WQ + kPanel, kHalfPanel, mb);
          bulk_g2s(dst + 2 * kT2 + (R::KE - kT2), src + R::KE, kTail, mb);
        }
      }
      if (!vzero) {
        const int lc = min(kC, rg.len - (c0 + ci) * kC);
        constexpr int kVec = DV / 8;
#pragma unroll 4
        for (int idx = lane; idx < 64 * kVec; idx += 32) {
          const int t = idx / kVec, cv = idx % kVec;
          const bool ok = t < lc;
          const __nv_bfloat16* src = ok ? vg + ((int64_t)(c0 + ci) * kC + t) * a.v.st + 8 * cv : vg;
          cp_async16(sbase + L::VT + b * 64 * L::kPitch * 2 + sw128(t, 8 * cv, 64), src, ok ? 16u : 0u);
        }
      }
      cp_async_mbar_arrive(mb);
    }
    cp_async_wait_all();
    // the bulk copies issued last into each buffer have landed (the phase they
    // complete is that barrier's latest), so none writes shared memory after exit
#pragma unroll
    for (int b = 0; b < 2; ++b)
      if (last[b] >= 0 && !mbar_wait(mbar_rec0 + 8 * b, (uint32_t)((last[b] >> 1) & 1), wait_limit))
        atomicOr(a.err, kErrTimeout);
  } else if (warp == 4) {
    // ======================= MMA warp =======================
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      const uint32_t rec = sbase + L::REC + b * L::kRecBuf;  // T2 at +0, zero tile, then the rest
      const uint32_t rWQ = rec + 2 * kT2 + (R::WQ - kT2);
      const uint32_t rAQ = rec + 2 * kT2 + (R::AQ - kT2);
      const uint32_t rKE = rec + 2 * kT2 + (R::KE - kT2);
      const uint32_t vt = sbase + L::VT + b * 64 * L::kPitch * 2;
      wait(mbar_rec0 + 8 * b, (ci >> 1) & 1);
      // U/O buffer b was last used by chunk ci - 2: its output must have been read out
      if (ci >= 2) wait(mbar_orel0 + 8 * b, (uint32_t)(((ci - 2) >> 1) & 1));
      // [U ; Q+ S] = [T_beta | -W ; 0 | Q+] [V ; S]; the V half needs no state, so it
      // is issued before the state's bf16 copy is ready
      if (lane == 0 && !*sFlag && !vzero) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tX(b), desc_kmajor(rec, 64, ks), desc_mnmajor(vt, 64, ks),
                   idesc_bf16(128, DV, false, true), ks > 0);
      }
      __syncwarp();
      bar_sync(1, 160);
      if (lane == 0 && !*sFlag) {
        fence_after_sync();
        // without values the state product starts the accumulator (rows 64..127,
        // Q+ S, are only read for outputs)
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tX(b), desc_kmajor(rWQ, 128, ks), desc_mnmajor(sbase + L::SB, DK, ks),
                   idesc_bf16(128, DV, false, true), (vzero && ks == 0) ? 0u : 1u);
        mma_commit(mbar_a);
      }
      __syncwarp();
      bar_sync(2, 160);
      // S += K_end^T U  (the state chain), then O += A_Q U (rows 64..127 of buffer b)
      if (lane == 0 && !*sFlag) {
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tS, desc_mnmajor(rKE, 64, ks), desc_mnmajor(vt, 64, ks),
                   idesc_bf16(128, DV, true, true), 1u);
        mma_commit(mbar_s);
        if (outs)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tX(b), desc_kmajor(rAQ - 64 * 128, 64, ks), desc_mnmajor(vt, 64, ks),
                     idesc_bf16(128, DV, false, true), 1u);
        mma_commit(mbar_free0 + 8 * b);  // chunk ci's output is ready; its buffers are free
      }
      __syncwarp();
    }
    // every product issued has completed before TMEM is freed (after an abort some
    // may still run; otherwise they were all waited on and this returns at once)
    if (lane == 0) {
      mma_commit(mbar_done);
      if (!mbar_wait(mbar_done, 0, wait_limit)) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ======================= TMEM <-> memory warps =======================
    // rows 64..127 of chunk pc's U/O buffer -> out (warps 2-3).  The values are
    // read from TMEM first and the buffer is released at once (orel, when
    // `release`); each warp then turns its 32 rows around through a small
    // shared staging area so that every store instruction writes four whole
    // 128-byte lines.
    auto store_out = [&](int pc, bool release) {
      const int lc = min(kC, rg.len - (c0 + pc) * kC);
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
      constexpr int kPass = DV < 64 ? DV : 64;  // columns per pass through the staging rows
      constexpr int kCh = kPass / 8;            // 16-byte chunks of a row per pass
#pragma unroll
      for (int half = 0; half < DV / kPass; ++half) {
        __syncwarp();  // the previous pass has been read back
#pragma unroll
        for (int u = 0; u < kCh; ++u) {
          const float* f = reinterpret_cast<const float*>(r[(kPass * half + 8 * u) >> 5]) + ((8 * u) & 31);
          st_shared_v4(stage + lane * 144 + 16 * u, pack_bf16(a.scale * f[0], a.scale * f[1]),
                       pack_bf16(a.scale * f[2], a.scale * f[3]), pack_bf16(a.scale * f[4], a.scale * f[5]),
                       pack_bf16(a.scale * f[6], a.scale * f[7]));
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < kCh; ++it) {
          const int rr = (32 / kCh) * it + lane / kCh, ch = lane % kCh;
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(stage + rr * 144 + 16 * ch));
          const int t = row0 + rr;
          if (t < lc)
            *reinterpret_cast<uint4*>(og + ((int64_t)(c0 + pc) * kC + t) * a.out_st + kPass * half + 8 * ch) = w;
        }
      }
    };
    for (int ci = 0; ci < nch; ++ci) {
      const int b = ci & 1;
      const uint32_t rec = sbase + L::REC + b * L::kRecBuf;
      const uint32_t vt = sbase + L::VT + b * 64 * L::kPitch * 2;
      // (1) bf16 copy of the state entering this chunk (read once from TMEM, kept in registers)
      uint32_t r[DV / 32][32];
      if (ci > 0) wait(mbar_s, (uint32_t)((ci - 1) & 1));
      if (tid < DK) {
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) tmem_ld32_async(tS + lane_base + 32 * q, r[q]);
        tmem_wait_ld();
        // prefix-cache checkpoint: the state after (c0 + ci) * 64 tokens of the sequence
        const int tok = (c0 + ci) * kC;
        if (a.ckpt && outs && tok > 0 && tok % a.ck_tokens == 0 && tok / a.ck_tokens <= a.ck_count) {
          float* dst = a.ckpt + ((int64_t)n * a.ck_count + tok / a.ck_tokens - 1) * a.ck_sr + h * a.ck_sh +
                       (int64_t)tid * a.dv + un.col;
#pragma unroll
          for (int q = 0; q < DV / 32; ++q)
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + 32 * q + i) =
                  make_float4(__uint_as_float(r[q][i]), __uint_as_float(r[q][i + 1]), __uint_as_float(r[q][i + 2]),
                              __uint_as_float(r[q][i + 3]));
        }
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
      // (2) decay the TMEM state by e^{G_C} of this chunk (overlaps the first product);
      // the state is read from TMEM again rather than kept in registers across the
      // record wait (217 instead of 255 registers at 128 columns, no spills)
      wait(mbar_rec0 + 8 * b, (ci >> 1) & 1);
      if (tid < DK) {
        const float pc = reinterpret_cast<const float*>(smem + (rec - sbase) + 2 * kT2 + (R::P - kT2))[tid];
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) tmem_ld32_async(tS + lane_base + 32 * q, r[q]);
        tmem_wait_ld();
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
        if (outs) {
          store_out(ci - 1, true);
        } else {  // no outputs: release the buffer at once
          fence_before_sync();
          mbar_arrive(mbar_orel0 + 8 * ((ci - 1) & 1));
        }
      }
    }
    // last output and the final state
    if (nch > 0) {
      wait(mbar_s, (uint32_t)((nch - 1) & 1));
      if (warp >= 2 && outs) {
        wait(mbar_free0 + 8 * ((nch - 1) & 1), (uint32_t)(((nch - 1) >> 1) & 1));
        store_out(nch - 1, false);
      }
    }
    // a checkpoint that falls on the sequence's end is the state after the last chunk
    const int end_tok = un.c1 * kC;
    const bool end_ck = a.ckpt && outs && nch > 0 && rg.len == end_tok && end_tok % a.ck_tokens == 0 &&
                        end_tok / a.ck_tokens <= a.ck_count;
    if ((un.fin || end_ck) && tid < DK) {
      float* dst = un.fin ? un.fin + (int64_t)tid * un.fin_ld : nullptr;
      float* cdst = end_ck ? a.ckpt + ((int64_t)n * a.ck_count + end_tok / a.ck_tokens - 1) * a.ck_sr +
                                 h * a.ck_sh + (int64_t)tid * a.dv + un.col
                           : nullptr;
#pragma unroll
      for (int cb = 0; cb < DV; cb += 32) {
        float v[32];
        tmem_ld32(tS + lane_base + cb, v);
        if (dst && cb < un.fin_cols) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + cb + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        if (cdst) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(cdst + cb + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------
// chunk offsets of each sequence (varlen): off[n] = sum_{m < n} ceil(len_m / 64),
// capped at `total` so no record index can fall outside the workspace; and, when
// soff is given, tail-segment offsets soff[n] = sum_{m < n} (segments_m - 1),
// capped at `ntail`
__global__ void kda_chunk_offsets_kernel(PrefillArgs a, int total, int* off, int* soff, int ntail) {
  __shared__ int part[256], spart[256];
  const int N = a.N;
  const int per = (N + 255) / 256;
  const int n0 = threadIdx.x * per;
  int s = 0, ss = 0;
  for (int i = 0; i < per; ++i) {
    const int n = n0 + i;
    if (n < N) {
      const int nc = (seq_range(a, n).len + kC - 1) / kC;
      s += nc;
      ss += num_segments(nc) - 1;
    }
  }
  part[threadIdx.x] = s;
  spart[threadIdx.x] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0, srun = 0;
    for (int i = 0; i < 256; ++i) {
      const int x = part[i], y = spart[i];
      part[i] = run;
      spart[i] = srun;
      run += x;
      srun += y;
    }
    off[N] = min(run, total);
    if (soff) soff[N] = min(srun, ntail);
  }
  __syncthreads();
  int run = part[threadIdx.x], srun = spart[threadIdx.x];
  for (int i = 0; i < per; ++i) {
    const int n = n0 + i;
    if (n < N) {
      const int nc = (seq_range(a, n).len + kC - 1) / kC;
      off[n] = min(run, total);
      if (soff) soff[n] = min(srun, ntail);
      run += nc;
      srun += num_segments(nc) - 1;
    }
  }
}

// ---------------------------------------------------------------------------
// States entering the tail segments: S_in(s + 1) = M_s S_in(s) + S~_s, in fp32,
// in order over the segments of each (sequence, head).  S_in(1) is segment 0's
// final state (serial pass 0).  One CTA per (sequence, head, 32 value columns).
constexpr int kCombineThreads = 256;
template <int DK>
struct CombineSmem {
  static constexpr int kMd = DK + 4;  // fp32 row stride of M
  static constexpr int kBytes = (DK * kMd + DK * 32) * 4;
};

template <int DK>
__global__ void __launch_bounds__(kCombineThreads) kda_segment_combine_kernel(PrefillArgs a, Split sp, Seg sg) {
  constexpr int RPT = DK / 32;  // rows per thread: 8 threads x 4 columns cover 32 columns
  using CS = CombineSmem<DK>;
  extern __shared__ float csm[];
  float* Ms = csm;                 // M: [DK][kMd]
  float* Ss = csm + DK * CS::kMd;  // state block: [DK][32]
  const int ncb = a.dv / 32;
  const int cb = blockIdx.x % ncb, nh = blockIdx.x / ncb;
  const int n = nh / a.H, h = nh - (nh / a.H) * a.H;
  const Range rg = seq_range(a, n);
  const int nc = min(num_chunks(sp, n), (rg.len + kC - 1) / kC);
  const int ns = num_segments(nc);
  if (ns < 3) return;
  const int t0 = tail_first(sg, n);
  if (t0 + ns - 2 >= tail_count(sg, a.N)) return;
  const int tid = threadIdx.x;
  const int r0 = RPT * (tid >> 3), cq = 4 * (tid & 7);
  const int64_t ldt = a.dv + DK;
  const float* sin0 = sg.sin + ((int64_t)t0 * a.H + h) * DK * a.dv + 32 * cb;
  for (int i = tid; i < DK * 8; i += kCombineThreads) {
    const int r = i >> 3, c = 4 * (i & 7);
    *reinterpret_cast<float4*>(Ss + r * 32 + c) = *reinterpret_cast<const float4*>(sin0 + (int64_t)r * a.dv + c);
  }
  for (int sgi = 2; sgi < ns; ++sgi) {
    // (S~ | M) of segment sgi - 1
    const float* tr = sg.tr + ((int64_t)(t0 + sgi - 2) * a.H + h) * DK * ldt;
    for (int i = tid; i < DK * DK / 4; i += kCombineThreads) {
      const int r = i / (DK / 4), k = 4 * (i % (DK / 4));
      *reinterpret_cast<float4*>(Ms + r * CS::kMd + k) = *reinterpret_cast<const float4*>(tr + r * ldt + a.dv + k);
    }
    __syncthreads();
    float acc[RPT][4];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(tr + (int64_t)(r0 + i) * ldt + 32 * cb + cq);
      acc[i][0] = x.x;
      acc[i][1] = x.y;
      acc[i][2] = x.z;
      acc[i][3] = x.w;
    }
#pragma unroll 4
    for (int k = 0; k < DK; ++k) {
      const float4 b = *reinterpret_cast<const float4*>(Ss + k * 32 + cq);
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float m = Ms[(r0 + i) * CS::kMd + k];
        acc[i][0] = fmaf(m, b.x, acc[i][0]);
        acc[i][1] = fmaf(m, b.y, acc[i][1]);
        acc[i][2] = fmaf(m, b.z, acc[i][2]);
        acc[i][3] = fmaf(m, b.w, acc[i][3]);
      }
    }
    __syncthreads();
    float* dst = sg.sin + ((int64_t)(t0 + sgi - 1) * a.H + h) * DK * a.dv + 32 * cb;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 x = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(Ss + (r0 + i) * 32 + cq) = x;
      *reinterpret_cast<float4*>(dst + (int64_t)(r0 + i) * a.dv + cq) = x;
    }
    __syncthreads();
  }
}


template <int DK>
constexpr int rec_bytes() { return Rec<DK>::kBytes; }

int64_t split_total_chunks(const PrefillArgs& a) {
  const int64_t nck = ((int64_t)a.T + kC - 1) / kC;
  return a.cu_seqlens ? nck + a.N : nck * a.N;
}

// Workspace plan: [chunk offsets | tail-segment offsets | records | (S~ | M) | S_in]
struct Plan {
  int64_t off_bytes, soff_bytes, rec_bytes, tr_bytes, sin_bytes;
  int ntail, tps;
  int64_t total() const { return off_bytes + soff_bytes + rec_bytes + tr_bytes + sin_bytes; }
};

Plan plan(const PrefillArgs& a) {
  Plan p{};
  const int64_t total = split_total_chunks(a);
  const int64_t nck = ((int64_t)a.T + kC - 1) / kC;
  p.off_bytes = a.cu_seqlens ? (((int64_t)(a.N + 1) * 4 + 1023) & ~int64_t(1023)) : 0;
  p.rec_bytes = total * a.H * (a.dk == 128 ? Rec<128>::kBytes : Rec<64>::kBytes);
  if (a.cu_seqlens) {
    // sum over sequences of (segments - 1) <= (sum of chunks) / kTailSeg: a
    // sequence of nc > kFirstSeg chunks has ceil((nc - kFirstSeg) / kTailSeg)
    // tail segments, at most nc / kTailSeg as kTailSeg <= kFirstSeg
    p.ntail = (int)(total / kTailSeg);
    p.tps = 0;
    p.soff_bytes = p.ntail ? (((int64_t)(a.N + 1) * 4 + 1023) & ~int64_t(1023)) : 0;
  } else {
    p.tps = num_segments((int)nck) - 1;
    p.ntail = a.N * p.tps;
    p.soff_bytes = 0;
  }
  p.tr_bytes = (int64_t)p.ntail * a.H * a.dk * (a.dv + a.dk) * 4;
  p.sin_bytes = (int64_t)p.ntail * a.H * a.dk * a.dv * 4;
  return p;
}

template <int DK, int DV>
cudaError_t launch(const PrefillArgs& a, void* ws, cudaStream_t s) {
  const Plan pl = plan(a);
  unsigned char* base = static_cast<unsigned char*>(ws);
  Split sp;
  sp.off = a.cu_seqlens ? reinterpret_cast<const int*>(base) : nullptr;
  sp.rec = base + pl.off_bytes + pl.soff_bytes;
  sp.total = (int)split_total_chunks(a);
  sp.nck = (int)(((int64_t)a.T + kC - 1) / kC);
  Seg sg;
  sg.soff = pl.soff_bytes ? reinterpret_cast<const int*>(base + pl.off_bytes) : nullptr;
  sg.tr = reinterpret_cast<float*>(sp.rec + pl.rec_bytes);
  sg.sin = reinterpret_cast<float*>(sp.rec + pl.rec_bytes + pl.tr_bytes);
  sg.ntail = pl.ntail;
  sg.tps = pl.tps;
  cudaError_t e;
  if (a.cu_seqlens) {
    launch_begin(s);
    kda_chunk_offsets_kernel<<<1, 256, 0, s>>>(a, sp.total, reinterpret_cast<int*>(base),
                                               sg.soff ? reinterpret_cast<int*>(base + pl.off_bytes) : nullptr,
                                               pl.ntail);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  auto prep = a.gate ? kda_chunk_prep_kernel<DK, true> : kda_chunk_prep_kernel<DK, false>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, PrepSmem<DK>::kAlloc);
  if (e != cudaSuccess) return e;
  // Value-column slices: d_v is split into 32- or 64-column CTAs, as finely as the
  // first pass's CTAs then still fit on the SMs at once, so that more SMs carry the
  // serial loop and each chunk step moves less.  Every slice CTA reads the whole
  // chunk record.  The first pass holds every sequence's first segment and, per tail
  // segment and head, the DV + DK augmented columns; the tail count is exact for
  // fixed-length batches and, with cu_seqlens, a lower bound from the total chunks.
  constexpr int DVM = DV == 128 ? 64 : DV;
  const int64_t nh = (int64_t)a.N * a.H;
  const int64_t tails = a.cu_seqlens ? std::max<int64_t>(0, (int64_t)sp.total - (int64_t)a.N * kFirstSeg) / kTailSeg
                                     : (int64_t)a.N * pl.tps;
  auto first_pass_ctas = [&](int w) { return nh * (DV / w) + tails * a.H * ((DV + DK + w - 1) / w); };
  const int W = first_pass_ctas(32) <= sm_count() ? 32 : (DVM != DV && first_pass_ctas(DVM) <= sm_count()) ? DVM : DV;
  // the second pass runs the tail segments alone: its own slice width (from the
  // workspace's tail-unit bound, which is exact for fixed-length batches)
  auto second_pass_ctas = [&](int w) { return (int64_t)pl.ntail * a.H * (DV / w); };
  const int W1 = second_pass_ctas(32) <= sm_count() ? 32 : (DVM != DV && second_pass_ctas(DVM) <= sm_count()) ? DVM : DV;
  using SerFn = void (*)(PrefillArgs, Split, Seg, int);
  auto ser_fn = [&](int w) -> SerFn {
    return w == 32 ? kda_chunk_serial_kernel<DK, 32> : w == DVM ? kda_chunk_serial_kernel<DK, DVM> : kda_chunk_serial_kernel<DK, DV>;
  };
  auto ser_bytes = [&](int w) {
    return w == 32 ? SerialSmem<DK, 32>::kAlloc : w == DVM ? SerialSmem<DK, DVM>::kAlloc : SerialSmem<DK, DV>::kAlloc;
  };
  const SerFn ser = ser_fn(W), ser1 = ser_fn(W1);
  const int ser_smem = ser_bytes(W), ser1_smem = ser_bytes(W1);
  e = cudaFuncSetAttribute(ser, cudaFuncAttributeMaxDynamicSharedMemorySize, ser_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ser1, cudaFuncAttributeMaxDynamicSharedMemorySize, ser1_smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)sp.total * a.H;
  const int grid = (int)(items < 2 * sm_count() ? items : 2 * sm_count());
  if (grid > 0) {
    launch_begin(s);
    prep<<<grid, kThreads, PrepSmem<DK>::kAlloc, s>>>(a, sp);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  // pass 0: every sequence's first segment, and the tail segments' (S~ | M).
  // Programmatic serialization lets its CTAs start while prep finishes.
  const int64_t nfirst = (int64_t)a.N * a.H * (DV / W);
  const int64_t ntail_ctas = (int64_t)pl.ntail * a.H * ((DV + DK + W - 1) / W);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nfirst + ntail_ctas));
    cfg.blockDim = dim3(kSerialThreads);
    cfg.dynamicSmemBytes = (size_t)ser_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = grid > 0 ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    launch_begin(s);
    if ((e = cudaLaunchKernelEx(&cfg, ser, a, sp, sg, 0)) != cudaSuccess || (e = launch_end(s)) != cudaSuccess)
      return e;
  }
  if (pl.ntail == 0) return cudaSuccess;
  // states entering the tail segments (only sequences of three or more segments need it)
  if (a.cu_seqlens ? pl.ntail >= 2 : pl.tps >= 2) {
    auto comb = kda_segment_combine_kernel<DK>;
    e = cudaFuncSetAttribute(comb, cudaFuncAttributeMaxDynamicSharedMemorySize, CombineSmem<DK>::kBytes);
    if (e != cudaSuccess) return e;
    launch_begin(s);
    comb<<<dim3((unsigned)((int64_t)a.N * a.H * (DV / 32))), kCombineThreads, CombineSmem<DK>::kBytes, s>>>(a, sp, sg);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = launch_end(s)) != cudaSuccess) return e;
  }
  // pass 1: the tail segments from their input states, with outputs
  launch_begin(s);
  ser1<<<dim3((unsigned)second_pass_ctas(W1)), kSerialThreads, ser1_smem, s>>>(a, sp, sg, 1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

}  // namespace

// SM count of the current device, looked up once per device (concurrent first
// calls may both look it up; they store the same value).
int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> counts[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) cudaGetLastError();
    return c > 0 ? c : 1;
  }
  int c = counts[dev].load(std::memory_order_relaxed);
  if (c <= 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) cudaGetLastError();
    if (c <= 0) c = 1;
    counts[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

size_t chunk_prefill_workspace_bytes(const PrefillArgs& a) { return (size_t)plan(a).total(); }

cudaError_t launch_chunk_prefill_tc(const PrefillArgs& a, void* workspace, cudaStream_t s) {
  if (!a.bf16) return cudaErrorInvalidValue;
  if (a.dk == 128 && a.dv == 128) return launch<128, 128>(a, workspace, s);
  if (a.dk == 128 && a.dv == 64) return launch<128, 64>(a, workspace, s);
  if (a.dk == 64 && a.dv == 128) return launch<64, 128>(a, workspace, s);
  if (a.dk == 64 && a.dv == 64) return launch<64, 64>(a, workspace, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
