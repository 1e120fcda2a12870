// Chunked backward of the KDA core: the gradient kernel on the tensor cores
// (d_k = d_v = 128, bf16 inputs).
//
// Per (chunk, head) the kernel follows the derivation in kda_backward_chunk.cuh.
// Every contraction runs as tcgen05.mma with fp32 accumulators in tensor memory:
//
//   D1 = S [dO; dY]^T     lanes d, columns (i of dO | i of dY): (dO S^T)^T, (dY S^T)^T
//   D2 = X U^T            lanes d, columns i: (U X^T)^T
//   D3 = [dO; dY] U^T     lanes (i of dO | i of dY), columns j: dO U^T, dY U^T
//   R1, R2                lanes d, columns i: the row forms inside the chunk,
//                         sum_{j <= i} M_ij k_j e^{G_i - G_j} for M = M1, M2
//   CF_I                  lanes d, columns j: the column form of sub-block I,
//                         sum_{i in I} (M1_ij q_i + M2_ij k_i) e^{G_i - c_I}
//
// with M1 = scale Tril(dO U^T), M2 = -StrictTril(diag(beta) dY U^T).  With the
// key channel d on the 128 lanes all products have M = 128.  The exponent
// references of the intra-chunk forms are those of 16-token sub-blocks (g in
// [-5, 0] keeps every factor within e^{+-80}): the row form of rows in sub-block I
// uses k_j e^{r_I - G_j} for j < 16 (I + 1) (one operand version per I, at most 1 for
// earlier sub-blocks), the column form refers row i to the end c_I of its own
// sub-block, and one factor per output element restores the exponent.
//
// S, X, U, dY, M1, M2 and the exponent-scaled q and k are fp32, so each operand is
// split into bf16 halves x = x_hi + x_lo (x_hi = bf16(x), x_lo = bf16(x - x_hi)) and
// a product is taken as a_hi b_hi + a_lo b_hi + a_hi b_lo: three bf16 MMAs with a
// relative error near 2^-16.  q, k, v and dO are bf16 already.
//
// dbeta needs no product of its own:
//   dbeta_i = sum_v dY (V - K+ S - A U) = rowdot(dY, V) - rowdot(K+, dY S^T) - rowdot(A, dY U^T).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_backward_chunk.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;
using bwdc::ChunkBwdArgs;
using bwdc::kC;
using bwdc::kSB;
using bwdc::ld4;
using bwdc::ld4t;
using bwdc::st4;
using bwdc::zero4;

constexpr int kTcThreads = 256;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: D3 is read before R1 is written over it
constexpr uint32_t kD1 = 0, kD2 = 128, kD3 = 192, kR1 = 192, kR2 = 256, kCF = 320;
// first column of CF_I (16 (I + 1) columns each)
__device__ __forceinline__ uint32_t cf_col(int I) { return kCF + 8u * (uint32_t)(I * (I + 1)); }

// Byte offsets in the 1024-byte aligned dynamic shared memory.
struct GradTcSmem {
  // first products: bf16 tiles, 128-byte swizzle, 128 rows x K = 128 (two 16 KB panels)
  static constexpr uint32_t TS = 0;         // S hi, then X hi
  static constexpr uint32_t TS_LO = 32768;  // S lo, then X lo
  static constexpr uint32_t TB = 65536;     // [dO; dY hi]
  static constexpr uint32_t TL = 98304;     // [0; dY lo]
  static constexpr uint32_t TU = 131072;    // [U hi; U lo]
  static constexpr uint32_t OPS = 163840;
  // intra-chunk forms
  static constexpr uint32_t M1_HI = TL, M1_LO = TL + 8192;  // 64 x 64 bf16 (rows i, columns j)
  static constexpr uint32_t M2_HI = TL + 16384, M2_LO = TL + 24576;
  // k e^{r_I - G}: version I, 16 (I + 1) rows x 128 (kr_hi / kr_lo)
  static constexpr uint32_t QC_HI = 0, QC_LO = 16384, KC_HI = 32768, KC_LO = 49152;  // 64 rows x 128
  static constexpr uint32_t KRAW = TB, QRAW = TB + 16384;  // k, q of the chunk: [64][128] bf16 rows
  static constexpr uint32_t DG = 0;  // [64][128] fp32 dG
  // kept throughout
  static constexpr uint32_t G = OPS;                  // [64][128] fp32 cumulative log-decay
  static constexpr uint32_t RR = G + 64 * 128 * 4;    // [5][128] r_0..r_3, G_C (c_I = r_{I+1})
  static constexpr uint32_t BETA = RR + 5 * 128 * 4;  // [64]
  static constexpr uint32_t GS = BETA + 64 * 4;       // [128] rowsum(S X)
  static constexpr int PB = 8;                        // dbeta partials per row (7 used)
  static constexpr uint32_t DBP = GS + 128 * 4;       // [64][PB]
  static constexpr uint32_t EKP = DBP + 64 * PB * 4;  // [2][128] sums of e k over half the rows
  static constexpr uint32_t PART = EKP + 2 * 128 * 4; // [128] scratch of the cumulative sum
  static constexpr uint32_t MBAR = PART + 128 * 4;    // four mbarriers
  static constexpr uint32_t SLOT = MBAR + 32;         // tensor-memory base address
  static constexpr uint32_t FLAG = SLOT + 4;          // a bounded wait gave up
  static constexpr uint32_t BYTES = SLOT + 16;
};
// Version I of k e^{r_I - G} (4096 (I + 1) bytes per half): the high halves fill
// [0, 40960), the low halves of versions 0..2 [40960, 65536) and that of version 3
// the U tile.  All are written after D2 has read the X and U tiles.
__device__ __forceinline__ uint32_t kr_hi(int I) { return 2048u * (uint32_t)(I * (I + 1)); }
__device__ __forceinline__ uint32_t kr_lo(int I) { return I < 3 ? 40960u + kr_hi(I) : GradTcSmem::TU; }
static_assert(GradTcSmem::KRAW >= 65536 && GradTcSmem::QRAW + 16384 <= GradTcSmem::M1_HI, "raw k, q between");
// dbeta partials of a row: [0, 4) -rowdot(K+, dY S^T) by lane quarter, [4, 6)
// -rowdot(A, dY U^T) by column half, [6] rowdot(dY, V)
constexpr int kDbAY = 4, kDbYV = 6, kDbCount = 7;

__device__ __forceinline__ uint32_t bf2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float bflo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bfhi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// x = hi + lo for a pair: returns hi, sets lo
__device__ __forceinline__ uint32_t split2(float a, float b, uint32_t& lo) {
  const uint32_t h = bf2(a, b);
  lo = bf2(a - bflo(h), b - bfhi(h));
  return h;
}

// hi and lo quadruples of x, stored 8 bytes each
__device__ __forceinline__ void store_split4(uint32_t hi_addr, uint32_t lo_addr, float4 x) {
  uint32_t l0, l1;
  const uint32_t h0 = split2(x.x, x.y, l0), h1 = split2(x.z, x.w, l1);
  asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(hi_addr), "r"(h0), "r"(h1) : "memory");
  asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(lo_addr), "r"(l0), "r"(l1) : "memory");
}

// the four values hi + lo stored by store_split4 at these addresses
__device__ __forceinline__ float4 load_split4(uint32_t hi_addr, uint32_t lo_addr) {
  uint32_t h0, h1, l0, l1;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(h0), "=r"(h1) : "r"(hi_addr) : "memory");
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(l0), "=r"(l1) : "r"(lo_addr) : "memory");
  float4 r;
  r.x = bflo(h0) + bflo(l0);
  r.y = bfhi(h0) + bfhi(l0);
  r.z = bflo(h1) + bflo(l1);
  r.w = bfhi(h1) + bfhi(l1);
  return r;
}

// eight bf16 at a 16-byte aligned shared address, as fp32
__device__ __forceinline__ void bf8(uint32_t addr, float (&x)[8]) {
  uint32_t u0, u1, u2, u3;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3) : "r"(addr) : "memory");
  x[0] = bflo(u0), x[1] = bfhi(u0), x[2] = bflo(u1), x[3] = bfhi(u1);
  x[4] = bflo(u2), x[5] = bfhi(u2), x[6] = bflo(u3), x[7] = bfhi(u3);
}

// 8-byte global -> shared copy, zero-filled when src_bytes == 0
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Sums v[r] over the 32 lanes for eight r at once (a transposing butterfly, nine
// shuffles); returns the sum for r = 4 bit4 + 2 bit3 + bit2 of the lane index.
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float w4[4], w2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w4[k] = (b4 ? v[k + 4] : v[k]) + __shfl_xor_sync(0xffffffffu, b4 ? v[k] : v[k + 4], 16);
#pragma unroll
  for (int k = 0; k < 2; ++k)
    w2[k] = (b3 ? w4[k + 2] : w4[k]) + __shfl_xor_sync(0xffffffffu, b3 ? w4[k] : w4[k + 2], 8);
  float w = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
  w += __shfl_xor_sync(0xffffffffu, w, 2);
  w += __shfl_xor_sync(0xffffffffu, w, 1);
  return w;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// G, the cumulative sum of g down the chunk (g zero past `rows`), into sG [64][128],
// and the sub-block references r_0 .. r_3 and G_C into rr [5][128]: two threads per
// channel, 32 rows each summed in registers; part is a [128] scratch.  All threads of
// the CTA call it; sG and rr are complete after the caller's next barrier.
__device__ __forceinline__ void chunk_cumsum(const float* gb, int64_t gst, int rows, float* sG, float* rr,
                                             float* part, int tid) {
  const int d = tid & 127, hf = tid >> 7;
  float g[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int r = 32 * hf + i;
    g[i] = r < rows ? gb[(int64_t)r * gst + d] : 0.f;
  }
#pragma unroll
  for (int i = 1; i < 32; ++i) g[i] += g[i - 1];
  if (hf == 0) part[d] = g[31];
  __syncthreads();
  const float off = hf ? part[d] : 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) sG[(32 * hf + i) * 128 + d] = g[i] + off;
  if (hf == 0) {
    rr[d] = 0.f;
    rr[128 + d] = g[15];
    rr[256 + d] = g[31];
  } else {
    rr[384 + d] = g[15] + off;
    rr[512 + d] = g[31] + off;
  }
}

// K = 128 (eight 16-deep steps) of one K-major product into the accumulator at d_tmem
__device__ __forceinline__ void mma_k128(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile, int b_row0,
                                         uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16(d_tmem, desc_kmajor(a_tile, 128, ks), desc_kmajor(b_tile, 128, ks, b_row0), idesc,
             (accumulate || ks > 0) ? 1u : 0u);
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1) kda_bwd_grad_tc_kernel(ChunkBwdArgs ca) {
  constexpr int DK = 128, DV = 128, NT = kTcThreads;
  using SM = GradTcSmem;
  using R = bwdc::Rec<DK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int f = blockIdx.x, h = blockIdx.y;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  bwdc::ChunkLoc L;
  if (!bwdc::locate(ca, f, L)) return;  // uniform across the CTA
  const int rows = L.rows;
  const float* rec = ca.rec + ((int64_t)f * a.H + h) * R::SIZE;
  const float* stt = ca.st + ((int64_t)f * a.H + h) * R::SSIZE;
  const T* ob = static_cast<const T*>(ba.dout.ptr) + L.b * ba.dout.sb + L.t * ba.dout.st + (int64_t)h * ba.dout.sh;
  const T* vb = static_cast<const T*>(a.v.ptr) + L.b * a.v.sb + L.t * a.v.st + (int64_t)h * a.v.sh;
  const T* qb = static_cast<const T*>(a.q.ptr) + L.b * a.q.sb + L.t * a.q.st + (int64_t)h * a.q.sh;
  const T* kb = static_cast<const T*>(a.k.ptr) + L.b * a.k.sb + L.t * a.k.st + (int64_t)h * a.k.sh;
  const float* gb = static_cast<const float*>(a.g.ptr) + L.b * a.g.sb + L.t * a.g.st + (int64_t)h * a.g.sh;
  const float* bb = a.beta + L.b * a.beta_sb + L.t * a.beta_st + (int64_t)h * a.beta_sh;
  float* sG = reinterpret_cast<float*>(smem + SM::G);
  float* rr = reinterpret_cast<float*>(smem + SM::RR);
  float* sb = reinterpret_cast<float*>(smem + SM::BETA);
  float* gs = reinterpret_cast<float*>(smem + SM::GS);
  float* dbp = reinterpret_cast<float*>(smem + SM::DBP);
  float* ekp = reinterpret_cast<float*>(smem + SM::EKP);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + SM::FLAG);
  const uint32_t mbar1 = s0 + SM::MBAR, mbar2 = mbar1 + 8, mbar3 = mbar1 + 16, mbar4 = mbar1 + 24;
  const int q4 = warp & 3, half = warp >> 2;  // lane quarter and column (or row) half of this warp
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

  if (warp == 0) tmem_alloc(s0 + SM::SLOT, kTmemCols);
  if (tid == 0) {
    mbar_init(mbar1, 1);
    mbar_init(mbar2, 1);
    mbar_init(mbar3, 1);
    mbar_init(mbar4, 1);
    *sFlag = 0;
    fence_mbar_init();
  }

  // ---- operand tiles of the first products ----
  // S -> TS (hi), TS_LO (lo): row d = warp + 8 u, columns 4 lane ..
  {
    float4 x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = ld4(stt + R::S + (int64_t)(warp + 8 * u) * DV + 4 * lane);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const uint32_t o = sw128(warp + 8 * u, 4 * lane, 128);
      store_split4(s0 + SM::TS + o, s0 + SM::TS_LO + o, x[u]);
    }
  }
  // dY -> TB rows 64.. (hi), TL rows 64.. (lo); U -> TU rows 0.. (hi), 64.. (lo);
  // rowdot(dY, V); dO -> TB rows 0..; zeros in TL rows 0..63
  {
    float4 y[8], uu[8], vv[8];
    uint2 o2[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = warp + 8 * u;
      y[u] = ld4(stt + R::DY + (int64_t)i * DV + 4 * lane);
      uu[u] = ld4(stt + R::U + (int64_t)i * DV + 4 * lane);
      vv[u] = i < rows ? ld4t<T>(vb + (int64_t)i * a.v.st + 4 * lane) : zero4();
      o2[u] = i < rows ? *reinterpret_cast<const uint2*>(ob + (int64_t)i * ba.dout.st + 4 * lane) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = warp + 8 * u;
      store_split4(s0 + SM::TB + sw128(64 + i, 4 * lane, 128), s0 + SM::TL + sw128(64 + i, 4 * lane, 128), y[u]);
      store_split4(s0 + SM::TU + sw128(i, 4 * lane, 128), s0 + SM::TU + sw128(64 + i, 4 * lane, 128), uu[u]);
      asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(s0 + SM::TB + sw128(i, 4 * lane, 128)), "r"(o2[u].x),
                   "r"(o2[u].y)
                   : "memory");
      const float yv = warp_sum(y[u].x * vv[u].x + y[u].y * vv[u].y + y[u].z * vv[u].z + y[u].w * vv[u].w);
      if (lane == 0) dbp[i * SM::PB + kDbYV] = yv;
    }
    for (int idx = tid; idx < 1024; idx += NT)  // rows 0..63 of both panels
      st_shared_v4(s0 + SM::TL + (uint32_t)(idx >> 9) * 16384u + (uint32_t)(idx & 511) * 16u, 0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM::SLOT);
  if (tid == 0) {
    const uint32_t i128 = idesc_bf16(128, 128, false, false), i64 = idesc_bf16(128, 64, false, false);
    // D1 = S [dO; dY]^T;  D3 = [dO; dY] U^T
    mma_k128(tmem + kD1, s0 + SM::TS, s0 + SM::TB, 0, i128, false);
    mma_k128(tmem + kD1, s0 + SM::TS_LO, s0 + SM::TB, 0, i128, true);
    mma_k128(tmem + kD1 + 64, s0 + SM::TS, s0 + SM::TL, 64, i64, true);
    mma_k128(tmem + kD3, s0 + SM::TB, s0 + SM::TU, 0, i64, false);
    mma_k128(tmem + kD3, s0 + SM::TB, s0 + SM::TU, 64, i64, true);
    mma_k128(tmem + kD3, s0 + SM::TL, s0 + SM::TU, 0, i64, true);
    mma_commit(mbar1);
  }

  // ---- while they run: log-decays, beta, the sub-block references; X ----
  float4 x[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) x[u] = ld4(stt + R::X + (int64_t)(warp + 8 * u) * DV + 4 * lane);
  if (tid < kC) sb[tid] = tid < rows ? bb[(int64_t)tid * a.beta_st] : 0.f;
  chunk_cumsum(gb, a.g.st, rows, sG, rr, reinterpret_cast<float*>(smem + SM::PART), tid);
  if (!mbar_wait(mbar1, 0)) *sFlag = 1;
  __syncthreads();
  if (*sFlag) goto fail;
  fence_after_sync();
  // raw k and q rows of the chunk (zero past the last row), landing while X is split
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int idx = tid + u * NT, i = idx >> 5, c = idx & 31;
    const int ic = i < rows ? i : 0;
    const uint32_t o = (uint32_t)(i * 256 + 8 * c), n = i < rows ? 8u : 0u;
    cp_async8(s0 + SM::KRAW + o, kb + (int64_t)ic * a.k.st + 4 * c, n);
    cp_async8(s0 + SM::QRAW + o, qb + (int64_t)ic * a.q.st + 4 * c, n);
  }
  cp_async_commit();

  // ---- X -> TS, TS_LO (S is read back from its tiles for rowsum(S X) first); D2 ----
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int d = warp + 8 * u;
    const uint32_t o = sw128(d, 4 * lane, 128);
    const float4 sv = load_split4(s0 + SM::TS + o, s0 + SM::TS_LO + o);
    const float p = warp_sum(sv.x * x[u].x + sv.y * x[u].y + sv.z * x[u].z + sv.w * x[u].w);
    if (lane == 0) gs[d] = p;
    store_split4(s0 + SM::TS + o, s0 + SM::TS_LO + o, x[u]);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    fence_after_sync();
    const uint32_t i64 = idesc_bf16(128, 64, false, false);
    // D2 = X U^T
    mma_k128(tmem + kD2, s0 + SM::TS, s0 + SM::TU, 0, i64, false);
    mma_k128(tmem + kD2, s0 + SM::TS_LO, s0 + SM::TU, 0, i64, true);
    mma_k128(tmem + kD2, s0 + SM::TS, s0 + SM::TU, 64, i64, true);
    mma_commit(mbar2);
  }

  // ---- D3 -> M1 = scale Tril(dO U^T), M2 = -StrictTril(diag(beta) dY U^T) as bf16
  //      halves (rows i, columns j) over TL; -rowdot(A, dY U^T) ----
  {
    float v[32];
    tmem_ld32(tmem + lane_base + kD3 + 32 * half, v);
    const int ip = 32 * q4 + lane, j0 = 32 * half;
    const bool m2 = ip >= kC;
    const int i = m2 ? ip - kC : ip;
    const float be = sb[i];
    float ay = 0.f;
    if (m2) {
      const float* arow = rec + R::A + i * kC + j0;
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 av = ld4(arow + k);
        ay += av.x * v[k] + av.y * v[k + 1] + av.z * v[k + 2] + av.w * v[k + 3];
      }
      dbp[i * SM::PB + kDbAY + half] = -ay;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = j0 + k;
      v[k] = m2 ? (j < i ? -be * v[k] : 0.f) : (j <= i ? a.scale * v[k] : 0.f);
    }
    const uint32_t hi = s0 + (m2 ? SM::M2_HI : SM::M1_HI), lo = s0 + (m2 ? SM::M2_LO : SM::M1_LO);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) ph[e] = split2(v[8 * c + 2 * e], v[8 * c + 2 * e + 1], pl[e]);
      const uint32_t o = sw128(i, j0 + 8 * c, 64);
      st_shared_v4(hi + o, ph[0], ph[1], ph[2], ph[3]);
      st_shared_v4(lo + o, pl[0], pl[1], pl[2], pl[3]);
    }
  }
  if (!mbar_wait(mbar2, 0)) *sFlag = 1;
  cp_async_wait_all();
  fence_before_sync();
  __syncthreads();
  if (*sFlag) goto fail;

  // ---- row-form operand: version I of k e^{r_I - G}, rows j < 16 (I + 1), as an
  //      MN-major tile (K rows j, M = d) ----
  for (int idx = tid; idx < 2560; idx += NT) {
    const int I = idx < 256 ? 0 : idx < 768 ? 1 : idx < 1536 ? 2 : 3;
    const int rem = idx - 128 * I * (I + 1), j = rem >> 4, d0 = 8 * (rem & 15);
    float kv[8];
    bf8(s0 + SM::KRAW + j * 256 + 2 * d0, kv);
    const float4 g0 = ld4(sG + j * DK + d0), g1 = ld4(sG + j * DK + d0 + 4);
    const float4 r0 = ld4(rr + I * DK + d0), r1 = ld4(rr + I * DK + d0 + 4);
    const float y[8] = {kv[0] * __expf(r0.x - g0.x), kv[1] * __expf(r0.y - g0.y), kv[2] * __expf(r0.z - g0.z),
                        kv[3] * __expf(r0.w - g0.w), kv[4] * __expf(r1.x - g1.x), kv[5] * __expf(r1.y - g1.y),
                        kv[6] * __expf(r1.z - g1.z), kv[7] * __expf(r1.w - g1.w)};
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) ph[e] = split2(y[2 * e], y[2 * e + 1], pl[e]);
    const uint32_t o = sw128(j, d0, kSB * (I + 1));
    st_shared_v4(s0 + kr_hi(I) + o, ph[0], ph[1], ph[2], ph[3]);
    st_shared_v4(s0 + kr_lo(I) + o, pl[0], pl[1], pl[2], pl[3]);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    fence_after_sync();
    // R1, R2 at rows (columns) of sub-block I: sum over j < 16 (I + 1)
    const uint32_t idesc = idesc_bf16(128, 16, true, false);
    for (int I = 0; I < 4; ++I) {
      const int kr = kSB * (I + 1);
      for (int m = 0; m < 2; ++m) {
        const uint32_t d = tmem + (m ? kR2 : kR1) + kSB * I;
        const uint32_t bh = s0 + (m ? SM::M2_HI : SM::M1_HI), bl = s0 + (m ? SM::M2_LO : SM::M1_LO);
        for (int ks = 0; ks <= I; ++ks) {
          const uint64_t ah = desc_mnmajor(s0 + kr_hi(I), kr, ks);
          const uint64_t al = desc_mnmajor(s0 + kr_lo(I), kr, ks);
          const uint64_t bhd = desc_kmajor(bh, 64, ks, kSB * I), bld = desc_kmajor(bl, 64, ks, kSB * I);
          mma_bf16(d, ah, bhd, idesc, ks > 0 ? 1u : 0u);
          mma_bf16(d, al, bhd, idesc, 1u);
          mma_bf16(d, ah, bld, idesc, 1u);
        }
      }
    }
    mma_commit(mbar3);
  }

  // ---- column-form operands q e^{G - c_I}, k e^{G - c_I} (row i in sub-block I),
  //      formed while the row forms run and stored once they are done ----
  {
    uint32_t qh[4][4], ql[4][4], kh[4][4], kl[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = tid + u * NT, i = idx >> 4, d0 = 8 * (idx & 15), I = i / kSB;
      float qv[8], kv[8];
      bf8(s0 + SM::QRAW + i * 256 + 2 * d0, qv);
      bf8(s0 + SM::KRAW + i * 256 + 2 * d0, kv);
      const float4 g0 = ld4(sG + i * DK + d0), g1 = ld4(sG + i * DK + d0 + 4);
      const float4 c0 = ld4(rr + (I + 1) * DK + d0), c1 = ld4(rr + (I + 1) * DK + d0 + 4);
      const float ex[8] = {__expf(g0.x - c0.x), __expf(g0.y - c0.y), __expf(g0.z - c0.z), __expf(g0.w - c0.w),
                           __expf(g1.x - c1.x), __expf(g1.y - c1.y), __expf(g1.z - c1.z), __expf(g1.w - c1.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qh[u][e] = split2(qv[2 * e] * ex[2 * e], qv[2 * e + 1] * ex[2 * e + 1], ql[u][e]);
        kh[u][e] = split2(kv[2 * e] * ex[2 * e], kv[2 * e + 1] * ex[2 * e + 1], kl[u][e]);
      }
    }
    if (!mbar_wait(mbar3, 0)) *sFlag = 1;
    __syncthreads();
    if (*sFlag) goto fail;
    fence_after_sync();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = tid + u * NT, i = idx >> 4, d0 = 8 * (idx & 15);
      const uint32_t o = sw128(i, d0, kC);
      st_shared_v4(s0 + SM::QC_HI + o, qh[u][0], qh[u][1], qh[u][2], qh[u][3]);
      st_shared_v4(s0 + SM::QC_LO + o, ql[u][0], ql[u][1], ql[u][2], ql[u][3]);
      st_shared_v4(s0 + SM::KC_HI + o, kh[u][0], kh[u][1], kh[u][2], kh[u][3]);
      st_shared_v4(s0 + SM::KC_LO + o, kl[u][0], kl[u][1], kl[u][2], kl[u][3]);
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    fence_after_sync();
    // CF_I: columns j < 16 (I + 1), sum over i in sub-block I
    for (int I = 0; I < 4; ++I) {
      const uint32_t idesc = idesc_bf16(128, kSB * (I + 1), true, true);
      const uint32_t d = tmem + cf_col(I);
      const uint64_t qhd = desc_mnmajor(s0 + SM::QC_HI, kC, I), qld = desc_mnmajor(s0 + SM::QC_LO, kC, I);
      const uint64_t khd = desc_mnmajor(s0 + SM::KC_HI, kC, I), kld = desc_mnmajor(s0 + SM::KC_LO, kC, I);
      const uint64_t m1h = desc_mnmajor(s0 + SM::M1_HI, kC, I), m1l = desc_mnmajor(s0 + SM::M1_LO, kC, I);
      const uint64_t m2h = desc_mnmajor(s0 + SM::M2_HI, kC, I), m2l = desc_mnmajor(s0 + SM::M2_LO, kC, I);
      mma_bf16(d, qhd, m1h, idesc, 0u);
      mma_bf16(d, qld, m1h, idesc, 1u);
      mma_bf16(d, qhd, m1l, idesc, 1u);
      mma_bf16(d, khd, m2h, idesc, 1u);
      mma_bf16(d, kld, m2h, idesc, 1u);
      mma_bf16(d, khd, m2l, idesc, 1u);
    }
    mma_commit(mbar4);
  }
  if (!mbar_wait(mbar4, 0)) *sFlag = 1;
  __syncthreads();
  if (*sFlag) goto fail;
  fence_after_sync();

  // ---- per (i, d): dq, dk and dG (lanes d, rows of this warp's half) ----
  //   E = e^{G} = e^{G - r_J} e^{r_J},  e^{G_C - G} = e^{c_J - G} e^{G_C - c_J},
  //   e^{c_I - G} = e^{c_J - G} e^{c_I - c_J}: two exponentials per element
  {
    const int d = 32 * q4 + lane;
    const __nv_bfloat16* sk = reinterpret_cast<const __nv_bfloat16*>(smem + SM::KRAW);
    const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(smem + SM::QRAW);
    float* sDG = reinterpret_cast<float*>(smem + SM::DG);
    float ek = 0.f;
#pragma unroll 1
    for (int g8 = 0; g8 < 4; ++g8) {
      const int i0 = 32 * half + 8 * g8, J = i0 / kSB;
      const float rJ = rr[J * DK + d], cJ = rr[(J + 1) * DK + d];
      const float eR = __expf(rJ);
      float rho[4];  // e^{c_I - c_J}, zero for I < J
#pragma unroll
      for (int I = 0; I < 4; ++I) rho[I] = I >= J ? __expf(rr[(I + 1) * DK + d] - cJ) : 0.f;
      uint32_t pq[8], pk[8], pe[8], r1[8], r2[8], cf[4][8];
      tmem_ld8_async(tmem + lane_base + kD1 + i0, pq);
      tmem_ld8_async(tmem + lane_base + kD1 + 64 + i0, pk);
      tmem_ld8_async(tmem + lane_base + kD2 + i0, pe);
      tmem_ld8_async(tmem + lane_base + kR1 + i0, r1);
      tmem_ld8_async(tmem + lane_base + kR2 + i0, r2);
#pragma unroll
      for (int I = 0; I < 4; ++I) tmem_ld8_async(tmem + lane_base + cf_col(I) + i0, cf[I]);
      tmem_wait_ld();
      float kp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = i0 + e;
        const float G = sG[i * DK + d];
        const float fr = __expf(G - rJ), fc = __expf(cJ - G);
        const float E = fr * eR, Ee = fc * rho[3];
        float cs = 0.f;
#pragma unroll
        for (int I = 0; I < 4; ++I) cs += rho[I] * __uint_as_float(cf[I][e]);
        const float b = fc * cs;
        const float kv = __bfloat162float(sk[i * DK + d]), qv = __bfloat162float(sq[i * DK + d]);
        const float pkv = __uint_as_float(pk[e]);
        const float dq = a.scale * __uint_as_float(pq[e]) * E + fr * __uint_as_float(r1[e]);
        const float av = -sb[i] * pkv * E + fr * __uint_as_float(r2[e]);
        const float ev = __uint_as_float(pe[e]) * Ee;
        sDG[i * DK + d] = (av - b - ev) * kv + dq * qv;
        ek += ev * kv;
        kp[e] = kv * E * pkv;
        if (i < rows) {
          const int64_t t = L.t + i;
          ba.dq.ptr[L.b * ba.dq.sb + t * ba.dq.st + (int64_t)h * ba.dq.sh + d] = dq;
          ba.dk.ptr[L.b * ba.dk.sb + t * ba.dk.st + (int64_t)h * ba.dk.sh + d] = av + b + ev;
        }
      }
      const float w = reduce8(kp, lane);
      if ((lane & 3) == 0) dbp[(i0 + (lane >> 2)) * SM::PB + q4] = -w;
    }
    ekp[half * DK + d] = ek;
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  // ---- dg: reverse cumulative sum down the chunk plus the G_C terms; dbeta ----
  if (tid < DK) {
    const int d = tid;
    const float* sDG = reinterpret_cast<const float*>(smem + SM::DG);
    float run = __expf(rr[4 * DK + d]) * gs[d] + ekp[d] + ekp[DK + d];
    for (int i = rows - 1; i >= 0; --i) {
      run += sDG[i * DK + d];
      ba.dg.ptr[L.b * ba.dg.sb + (L.t + i) * ba.dg.st + (int64_t)h * ba.dg.sh + d] = run;
    }
  } else if (tid - DK < rows) {
    const int i = tid - DK;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kDbCount; ++q) acc += dbp[i * SM::PB + q];
    ba.dbeta[L.b * ba.db_sb + (L.t + i) * ba.db_st + (int64_t)h * ba.db_sh] = acc;
  }
  return;

fail:
  // a product did not complete in time: report it, give the tensor core a bounded
  // second wait for what was issued, free the tensor memory and leave
  if (tid == 0) {
    atomicOr(a.err, kErrTimeout);
    mbar_wait(mbar1, 0);
    mbar_wait(mbar2, 0);
    mbar_wait(mbar3, 0);
    mbar_wait(mbar4, 0);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// prep on the tensor cores: the state-independent chunk matrices of one (chunk,
// head), d_k = d_v = 128, bf16 inputs.  Records and their meaning are those of
// the fp32 prep (bwdc::Rec): W = T diag(beta) K+, K_end, U_bar = T diag(beta) V,
// e^{G_C}, W_y = T^T K_end, diag(beta) K+, V_y = scale T^T A_Q^T dO,
// Z_q = scale Q+^T dO, A = StrictTril(K+ K-^T).
//
//   Gram  D_G = [k e^{G - r_I}; q e^{G - r_I}] Y^T with the column versions
//         Y = [k e^{r_0 - G} (rows < 16); ...; k e^{r_3 - G} (rows < 64)]: lanes
//         (i of k | i of q), 160 columns; row i of sub-block I reads version I,
//         giving A = K+ K-^T and A_Q = Q+ K-^T with every factor within e^{+-80}
//   D_ZQ  = dO^T (scale Q+)     lanes v, columns d      (Z_q^T)
//   D_VT  = dO^T (scale A_Q)    lanes v, columns j      (V_t^T, V_t = scale A_Q^T dO)
//   D_W   = (diag(beta) K+)^T T^T   lanes d, columns i  (W^T)
//   D_WY  = K_end^T T               lanes d, columns i  (W_y^T)
//   D_UB  = (diag(beta) V)^T T^T    lanes v, columns i  (U_bar^T)
//   D_VY  = V_t^T T                 lanes v, columns i  (V_y^T)
//
// T = (I + diag(beta) A)^-1 is formed on the CUDA cores (invert_lower) while
// D_ZQ and D_VT run.  fp32 operands are split into bf16 halves as in the gradient
// kernel; dO is bf16 already.
//
// The record keeps the fp32 layout's offsets and sizes but holds what the
// tensor-core state passes load (RecTc): W and W_y as [hi; lo] bf16 tiles of 128
// rows x K = 128 (K-major), K_end and -diag(beta) K+ as hi and lo MN-major tiles
// (K rows j x 128 channels), U_bar, V_y and Z_q slice-major ([d_v / 32] slices of
// 32 columns; Z_q's 16-byte chunks of row d rotated by d), e^{G_C} and A as before.
struct PrepTcSmem {
  // Gram operands (bf16 halves, K = 128): X 128 rows, Y 160 rows
  static constexpr uint32_t XH = 0, XL = 32768, YH = 65536, YL = 106496;  // ends 147456
  // after the Gram
  static constexpr uint32_t AQH = 0, AQL = 8192;       // scale A_Q: 64 x 64, rows i
  static constexpr uint32_t DOT = 16384;               // dO: K rows i x 128 v (MN-major)
  static constexpr uint32_t QPH = 32768, QPL = 49152;  // scale Q+: K rows i x 128 d (MN-major)
  static constexpr int PA = 68;                        // row pitch of the fp32 matrices
  static constexpr uint32_t SA = 65536, SAQ = SA + 64 * PA * 4, STT = SAQ + 64 * PA * 4;  // fp32 A, A_Q, T
  static constexpr uint32_t B0 = STT + 64 * PA * 4;    // fp32 [16][64] scratch of the inverse
  static constexpr uint32_t TH = 147456, TL = 155648;  // T: 64 x 64, rows i
  // after D_ZQ, D_VT and the inverse
  static constexpr uint32_t BKH = 0, BKL = 16384;      // diag(beta) K+: K rows j x 128 d
  static constexpr uint32_t KEH = 32768, KEL = 49152;  // K_end: K rows j x 128 d
  static constexpr uint32_t BVH = 65536, BVL = 81920;  // diag(beta) V: K rows j x 128 v
  static constexpr uint32_t VTH = 98304, VTL = 114688; // V_t^T: 128 rows v x K = 64 j (K-major)
  static constexpr uint32_t OPS = 163840;
  static_assert(B0 + 16 * 64 * 4 <= TH && VTL + 16384 <= TH, "fp32 scratch and tiles stay below T");
  // kept throughout
  static constexpr uint32_t G = OPS;                  // [64][128] fp32 cumulative log-decay
  static constexpr uint32_t RR = G + 64 * 128 * 4;    // [5][128] r_0..r_3, G_C
  static constexpr uint32_t BETA = RR + 5 * 128 * 4;  // [64]
  static constexpr uint32_t PART = BETA + 64 * 4;     // [128] scratch of the cumulative sum
  static constexpr uint32_t MBAR = PART + 128 * 4;    // three mbarriers
  static constexpr uint32_t SLOT = MBAR + 24;
  static constexpr uint32_t FLAG = SLOT + 4;
  static constexpr uint32_t BYTES = SLOT + 16;
};
// tensor-memory columns (D_UB and D_VY reuse the Gram's after it has been read)
constexpr uint32_t kPG = 0, kPZQ = 160, kPVT = 288, kPW = 352, kPWY = 416, kPUB = 0, kPVY = 64;

// eight fp32 of shared memory at a 16-byte aligned address
__device__ __forceinline__ void lds8(const float* p, float (&x)[8]) {
  const float4 a = ld4(p), b = ld4(p + 4);
  x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
// eight values as bf16 halves into two tiles at byte offset o
__device__ __forceinline__ void store_split8(uint32_t hi, uint32_t lo, uint32_t o, const float (&x)[8]) {
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) ph[e] = split2(x[2 * e], x[2 * e + 1], pl[e]);
  st_shared_v4(hi + o, ph[0], ph[1], ph[2], ph[3]);
  st_shared_v4(lo + o, pl[0], pl[1], pl[2], pl[3]);
}
// eight bf16 of row i (zero past `rows`) at 8-byte aligned p
template <typename T>
__device__ __forceinline__ void row8(const T* base, int64_t st, int i, int rows, int d0, float (&x)[8]) {
  if (i < rows) {
    const float4 a = ld4t<T>(base + (int64_t)i * st + d0), b = ld4t<T>(base + (int64_t)i * st + d0 + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
  }
}

// eight values as bf16 halves into a pair of 16 KB global tiles (hi, then lo) at byte offset o
__device__ __forceinline__ void rec_split8(unsigned char* tile, uint32_t o, const float (&x)[8]) {
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) ph[e] = split2(x[2 * e], x[2 * e + 1], pl[e]);
  *reinterpret_cast<uint4*>(tile + o) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
  *reinterpret_cast<uint4*>(tile + 16384 + o) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
}

// eight bf16 of row i (zero past `rows`) as a raw uint4
template <typename T>
__device__ __forceinline__ uint4 raw8(const T* base, int64_t st, int i, int rows, int d0) {
  if (i >= rows) return make_uint4(0u, 0u, 0u, 0u);
  const uint2 a = *reinterpret_cast<const uint2*>(base + (int64_t)i * st + d0);
  const uint2 b = *reinterpret_cast<const uint2*>(base + (int64_t)i * st + d0 + 4);
  return make_uint4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void unpack8(uint4 u, float (&x)[8]) {
  x[0] = bflo(u.x), x[1] = bfhi(u.x), x[2] = bflo(u.y), x[3] = bfhi(u.y);
  x[4] = bflo(u.z), x[5] = bfhi(u.z), x[6] = bflo(u.w), x[7] = bfhi(u.w);
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1) kda_bwd_prep_tc_kernel(ChunkBwdArgs ca) {
  constexpr int DK = 128, DV = 128, NT = kTcThreads;
  using SM = PrepTcSmem;
  using R = bwdc::Rec<DK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int f = blockIdx.x, h = blockIdx.y;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  bwdc::ChunkLoc L;
  if (!bwdc::locate(ca, f, L)) return;  // uniform across the CTA
  const int rows = L.rows;
  float* rec = ca.rec + ((int64_t)f * a.H + h) * R::SIZE;
  const T* qb = static_cast<const T*>(a.q.ptr) + L.b * a.q.sb + L.t * a.q.st + (int64_t)h * a.q.sh;
  const T* kb = static_cast<const T*>(a.k.ptr) + L.b * a.k.sb + L.t * a.k.st + (int64_t)h * a.k.sh;
  const T* vb = static_cast<const T*>(a.v.ptr) + L.b * a.v.sb + L.t * a.v.st + (int64_t)h * a.v.sh;
  const T* ob = static_cast<const T*>(ba.dout.ptr) + L.b * ba.dout.sb + L.t * ba.dout.st + (int64_t)h * ba.dout.sh;
  const float* gb = static_cast<const float*>(a.g.ptr) + L.b * a.g.sb + L.t * a.g.st + (int64_t)h * a.g.sh;
  const float* bb = a.beta + L.b * a.beta_sb + L.t * a.beta_st + (int64_t)h * a.beta_sh;
  float* sG = reinterpret_cast<float*>(smem + SM::G);
  float* rr = reinterpret_cast<float*>(smem + SM::RR);
  float* sb = reinterpret_cast<float*>(smem + SM::BETA);
  float* sA = reinterpret_cast<float*>(smem + SM::SA);
  float* sAQ = reinterpret_cast<float*>(smem + SM::SAQ);
  float* sT = reinterpret_cast<float*>(smem + SM::STT);
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + SM::FLAG);
  const uint32_t mbarG = s0 + SM::MBAR, mbar2 = mbarG + 8, mbar1 = mbarG + 16;
  const int q4 = warp & 3, half = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const float scale = a.scale;

  if (warp == 0) tmem_alloc(s0 + SM::SLOT, kTmemCols);
  if (tid == 0) {
    mbar_init(mbarG, 1);
    mbar_init(mbar2, 1);
    mbar_init(mbar1, 1);
    *sFlag = 0;
    fence_mbar_init();
  }
  // This thread's rows (tid >> 4) + 16 u (one in each sub-block u) and channels
  // d0 .. d0 + 7 of k, q, v and dO, loaded once; every elementwise step below uses
  // this mapping.
  const int r0 = tid >> 4, d0 = 8 * (tid & 15);
  uint4 kr[4], qr[4], vr[4], orw[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    kr[u] = raw8<T>(kb, a.k.st, r0 + 16 * u, rows, d0);
    qr[u] = raw8<T>(qb, a.q.st, r0 + 16 * u, rows, d0);
    vr[u] = raw8<T>(vb, a.v.st, r0 + 16 * u, rows, d0);
    orw[u] = raw8<T>(ob, ba.dout.st, r0 + 16 * u, rows, d0);
  }
  // ---- log-decays, beta; cumulative sums and the sub-block references ----
  if (tid < kC) sb[tid] = tid < rows ? bb[(int64_t)tid * a.beta_st] : 0.f;
  chunk_cumsum(gb, a.g.st, rows, sG, rr, reinterpret_cast<float*>(smem + SM::PART), tid);
  __syncthreads();
  // ---- Gram operands: X rows (k then q) referred to their sub-block start, and the
  //      column versions of k (row j of sub-block u appears in versions u .. 3) ----
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = r0 + 16 * u;
    float k8[8], q8[8], g[8], rv[8];
    unpack8(kr[u], k8);
    unpack8(qr[u], q8);
    lds8(sG + i * DK + d0, g);
    lds8(rr + u * DK + d0, rv);
    float x[8], y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float f = __expf(g[e] - rv[e]);
      x[e] = k8[e] * f;
      y[e] = q8[e] * f;
    }
    store_split8(s0 + SM::XH, s0 + SM::XL, sw128(i, d0, 128), x);
    store_split8(s0 + SM::XH, s0 + SM::XL, sw128(64 + i, d0, 128), y);
#pragma unroll
    for (int I = u; I < 4; ++I) {
      lds8(rr + I * DK + d0, rv);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = k8[e] * __expf(rv[e] - g[e]);
      store_split8(s0 + SM::YH, s0 + SM::YL, sw128(8 * I * (I + 1) + i, d0, 160), y);
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM::SLOT);
  if (tid == 0) {
    const uint32_t idg = idesc_bf16(128, 160, false, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t xh = desc_kmajor(s0 + SM::XH, 128, ks), xl = desc_kmajor(s0 + SM::XL, 128, ks);
      const uint64_t yh = desc_kmajor(s0 + SM::YH, 160, ks), yl = desc_kmajor(s0 + SM::YL, 160, ks);
      mma_bf16(tmem + kPG, xh, yh, idg, ks > 0 ? 1u : 0u);
      mma_bf16(tmem + kPG, xl, yh, idg, 1u);
      mma_bf16(tmem + kPG, xh, yl, idg, 1u);
    }
    mma_commit(mbarG);
  }
  // ---- while the Gram runs: the elementwise records K_end, -diag(beta) K+ (as tiles), e^{G_C} ----
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = r0 + 16 * u;
    float k8[8], g[8], gc[8], ke[8], kp[8];
    unpack8(kr[u], k8);
    lds8(sG + i * DK + d0, g);
    lds8(rr + 4 * DK + d0, gc);
    const float be = sb[i];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ke[e] = k8[e] * __expf(gc[e] - g[e]);
      kp[e] = be * k8[e] * __expf(g[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) kp[e] = -kp[e];
    const uint32_t o = sw128(i, d0, 64);
    rec_split8(reinterpret_cast<unsigned char*>(rec + R::KE), o, ke);
    rec_split8(reinterpret_cast<unsigned char*>(rec + R::KB), o, kp);
  }
  if (tid < DK) rec[R::EGC + tid] = __expf(rr[4 * DK + tid]);
  if (!mbar_wait(mbarG, 0)) *sFlag = 1;
  __syncthreads();
  if (*sFlag) goto fail;
  fence_after_sync();

  // ---- D_G -> A (strict) and A_Q (inclusive), fp32 ----
  for (int idx = tid; idx < 64 * SM::PA / 4; idx += NT) st4(sT + 4 * idx, zero4());  // T starts at zero
  {
    // warp quarter q4 holds rows 32 (q4 & 1) .. + 31 of k (q4 < 2) or q: sub-blocks
    // Ia (lanes 0-15) and Ia + 1 (lanes 16-31), whose versions are adjacent columns
    const int Ia = 2 * (q4 & 1), ca0 = 8 * Ia * (Ia + 1), na = kSB * (Ia + 1), nab = na + kSB * (Ia + 2);
    const int nchunk = nab / 16, c_lo = half ? (nchunk + 1) / 2 : 0, c_hi = half ? nchunk : (nchunk + 1) / 2;
    const int i = 32 * (q4 & 1) + lane;
    const bool qrow = q4 >= 2;
    float* dst = (qrow ? sAQ : sA) + i * SM::PA;
    for (int c = c_lo; c < c_hi; ++c) {
      float v[16];
      tmem_ld16(tmem + lane_base + kPG + ca0 + 16 * c, v);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int col = 16 * c + t;
        const int j = lane < 16 ? col : col - na;
        const bool mine = lane < 16 ? col < na : col >= na;
        if (mine) dst[j] = (qrow ? j <= i : j < i) ? v[t] : 0.f;
      }
    }
    // columns past this row's version (j >= 16 (I + 1) > i) are zero
    if (half) {
      const int jz = kSB * (i / kSB + 1);
      for (int j = jz; j < kC; j += 4) st4(dst + j, zero4());
    }
  }
  __syncthreads();
  // ---- record A; the operands of D_ZQ and D_VT ----
  for (int idx = tid; idx < kC * kC / 4; idx += NT) {
    const int i = idx >> 4, j4 = 4 * (idx & 15);
    st4(rec + R::A + i * kC + j4, ld4(sA + i * SM::PA + j4));
  }
  for (int idx = tid; idx < 512; idx += NT) {  // scale A_Q: rows i, octets of j
    const int i = idx >> 3, j0 = 8 * (idx & 7);
    float x[8];
    lds8(sAQ + i * SM::PA + j0, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= scale;
    store_split8(s0 + SM::AQH, s0 + SM::AQL, sw128(i, j0, 64), x);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {  // dO rows (exact) and scale Q+ rows
    const int i = r0 + 16 * u;
    const uint32_t o = sw128(i, d0, 64);
    st_shared_v4(s0 + SM::DOT + o, orw[u].x, orw[u].y, orw[u].z, orw[u].w);
    float x[8], g[8];
    unpack8(qr[u], x);
    lds8(sG + i * DK + d0, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= scale * __expf(g[e]);
    store_split8(s0 + SM::QPH, s0 + SM::QPL, o, x);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    fence_after_sync();
    const uint32_t izq = idesc_bf16(128, 128, true, true), ivt = idesc_bf16(128, 64, true, true);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t ad = desc_mnmajor(s0 + SM::DOT, kC, ks);
      mma_bf16(tmem + kPZQ, ad, desc_mnmajor(s0 + SM::QPH, kC, ks), izq, ks > 0 ? 1u : 0u);
      mma_bf16(tmem + kPZQ, ad, desc_mnmajor(s0 + SM::QPL, kC, ks), izq, 1u);
      mma_bf16(tmem + kPVT, ad, desc_mnmajor(s0 + SM::AQH, kC, ks), ivt, ks > 0 ? 1u : 0u);
      mma_bf16(tmem + kPVT, ad, desc_mnmajor(s0 + SM::AQL, kC, ks), ivt, 1u);
    }
    mma_commit(mbar2);
  }
  // ---- T = (I + diag(beta) A)^-1 on the CUDA cores meanwhile; its bf16 halves ----
  bwdc::invert_lower<NT>(sA, sT, sb, reinterpret_cast<float*>(smem + SM::B0), SM::PA, 64, tid);
  for (int idx = tid; idx < 512; idx += NT) {
    const int i = idx >> 3, j0 = 8 * (idx & 7);
    float x[8];
    lds8(sT + i * SM::PA + j0, x);
    store_split8(s0 + SM::TH, s0 + SM::TL, sw128(i, j0, 64), x);
  }
  if (!mbar_wait(mbar2, 0)) *sFlag = 1;
  __syncthreads();
  if (*sFlag) goto fail;
  fence_after_sync();
  // ---- D_VT -> V_t^T halves (rows v, K = j); D_ZQ -> record Z_q [d][v] ----
  {
    const int v = 32 * q4 + lane;
    float x[32];
    tmem_ld32(tmem + lane_base + kPVT + 32 * half, x);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[8 * c + e];
      store_split8(s0 + SM::VTH, s0 + SM::VTL, sw128(v, 32 * half + 8 * c, 128), y);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tmem_ld32(tmem + lane_base + kPZQ + 64 * half + 32 * c, x);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int dd = 64 * half + 32 * c + k;  // row d of slice v / 32; chunk (v % 32) / 4 rotated by d
        rec[R::ZQ + (v >> 5) * (DK * 32) + dd * 32 + ((((v & 31) >> 2) + dd) & 7) * 4 + (v & 3)] = x[k];
      }
    }
  }
  // ---- operands of the T products: diag(beta) K+, K_end, diag(beta) V (rows j) ----
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int j = r0 + 16 * u;
    const uint32_t o = sw128(j, d0, 64);
    float x[8], g[8], gc[8], y[8];
    unpack8(kr[u], x);
    lds8(sG + j * DK + d0, g);
    lds8(rr + 4 * DK + d0, gc);
    const float be = sb[j];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      y[e] = be * x[e] * __expf(g[e]);
      x[e] *= __expf(gc[e] - g[e]);
    }
    store_split8(s0 + SM::BKH, s0 + SM::BKL, o, y);
    store_split8(s0 + SM::KEH, s0 + SM::KEL, o, x);
    unpack8(vr[u], x);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= be;
    store_split8(s0 + SM::BVH, s0 + SM::BVL, o, x);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    fence_after_sync();
    const uint32_t ik = idesc_bf16(128, 64, true, false), im = idesc_bf16(128, 64, true, true);
    const uint32_t iv = idesc_bf16(128, 64, false, true);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t tkh = desc_kmajor(s0 + SM::TH, 64, ks), tkl = desc_kmajor(s0 + SM::TL, 64, ks);
      const uint64_t tmh = desc_mnmajor(s0 + SM::TH, kC, ks), tml = desc_mnmajor(s0 + SM::TL, kC, ks);
      const uint64_t bkh = desc_mnmajor(s0 + SM::BKH, kC, ks), bkl = desc_mnmajor(s0 + SM::BKL, kC, ks);
      const uint64_t keh = desc_mnmajor(s0 + SM::KEH, kC, ks), kel = desc_mnmajor(s0 + SM::KEL, kC, ks);
      const uint64_t bvh = desc_mnmajor(s0 + SM::BVH, kC, ks), bvl = desc_mnmajor(s0 + SM::BVL, kC, ks);
      const uint64_t vth = desc_kmajor(s0 + SM::VTH, 128, ks), vtl = desc_kmajor(s0 + SM::VTL, 128, ks);
      const uint32_t acc = ks > 0 ? 1u : 0u;
      mma_bf16(tmem + kPW, bkh, tkh, ik, acc);
      mma_bf16(tmem + kPW, bkl, tkh, ik, 1u);
      mma_bf16(tmem + kPW, bkh, tkl, ik, 1u);
      mma_bf16(tmem + kPWY, keh, tmh, im, acc);
      mma_bf16(tmem + kPWY, kel, tmh, im, 1u);
      mma_bf16(tmem + kPWY, keh, tml, im, 1u);
      mma_bf16(tmem + kPUB, bvh, tkh, ik, acc);
      mma_bf16(tmem + kPUB, bvl, tkh, ik, 1u);
      mma_bf16(tmem + kPUB, bvh, tkl, ik, 1u);
      mma_bf16(tmem + kPVY, vth, tmh, iv, acc);
      mma_bf16(tmem + kPVY, vtl, tmh, iv, 1u);
      mma_bf16(tmem + kPVY, vth, tml, iv, 1u);
    }
    mma_commit(mbar1);
  }
  if (!mbar_wait(mbar1, 0)) *sFlag = 1;
  __syncthreads();
  if (*sFlag) goto fail;
  fence_after_sync();
  // ---- records W, W_y (lanes d: [hi; lo] tiles) and U_bar, V_y (lanes v: slice-major) ----
  {
    const int c = 32 * q4 + lane;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      float x[32];
      tmem_ld32(tmem + lane_base + (m ? kPWY : kPW) + 32 * half, x);
      unsigned char* t = reinterpret_cast<unsigned char*>(rec + (m ? R::WY : R::W));
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int i = 32 * half + k;
        uint32_t lo;
        const uint32_t hi = split2(x[k], 0.f, lo);
        *reinterpret_cast<uint16_t*>(t + sw128(i, c, 128)) = (uint16_t)hi;
        *reinterpret_cast<uint16_t*>(t + sw128(kC + i, c, 128)) = (uint16_t)lo;
      }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      float x[32];
      tmem_ld32(tmem + lane_base + (m ? kPVY : kPUB) + 32 * half, x);
      float* dst = rec + (m ? R::VY : R::UB) + (c >> 5) * (kC * 32) + (c & 31);
#pragma unroll
      for (int k = 0; k < 32; ++k) dst[(32 * half + k) * 32] = x[k];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  return;

fail:
  if (tid == 0) {
    atomicOr(a.err, kErrTimeout);
    mbar_wait(mbarG, 0);
    mbar_wait(mbar2, 0);
    mbar_wait(mbar1, 0);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// forward and reverse state passes on the tensor cores (d_k = d_v = 128, bf16
// inputs, records as the tensor-core prep writes them).  One CTA per (sequence,
// head, 32 value columns); the 32-column slice of the state lives in tensor memory
// (lanes d) and every chunk takes two products:
//   forward   D_U = [W_hi; W_lo] [S_hi | S_lo]   U  = U_bar - (sum of the four quarters)
//             S  <- e^{G_C} S + K_end^T U
//   reverse   D_U = [W_y,hi; W_y,lo] [X_hi | X_lo]  dY = V_y + (sum of the four quarters)
//             X  <- e^{G_C} X + Z_q + (-diag(beta) K+)^T dY,  dv = diag(beta) dY
// The bf16 halves of S (or X) and of U (or dY) sit side by side along N (N = 64), so a
// product of split operands takes one chain of N = 64 MMAs plus, for the state
// update, one chain of N = 32 (K_end,lo U_hi): 16 MMAs per chunk.  The state update's
// N = 64 chain leaves K_end,hi U_lo in columns 32..63 of the state accumulator,
// which are added in when the state is next read and then cleared.  The next
// chunk's record tiles (64 KB, and the reverse pass's 16 KB Z_q slice) arrive by bulk
// copy into the other buffer while this chunk runs; U_bar / V_y rows, e^{G_C} and
// beta are loaded into registers one chunk ahead.
struct PassTcSmem {
  static constexpr uint32_t BUF = 65536;     // two buffers: [W_hi; W_lo] tile, then K_end hi, lo tiles
  static constexpr uint32_t M1 = 32768;      // offset of the second matrix in a buffer
  static constexpr uint32_t ZQB = 2 * BUF;   // reverse: two Z_q slices, [128][32] fp32 (rotated chunks)
  static constexpr uint32_t SB = ZQB + 32768;  // state halves: K rows d (128) x [hi 32 | lo 32], MN-major
  static constexpr uint32_t UB = SB + 16384;   // U (or dY) halves: K rows i (64) x [hi 32 | lo 32]
  static constexpr int PX = 33;                // exchange rows: the low-half rows of D_U, [64][33] fp32
  static constexpr uint32_t XCH = UB + 8192;
  static constexpr uint32_t MBAR = XCH + 64 * PX * 4;  // rec0, rec1, u, s, done
  static constexpr uint32_t SLOT = MBAR + 40;
  static constexpr uint32_t FLAG = SLOT + 4;
  static constexpr uint32_t BYTES = SLOT + 16;
};
constexpr uint32_t kPassTmemCols = 128;  // state accumulator at 0 (64 columns), D_U at 64

template <bool REV>
__global__ void __launch_bounds__(kTcThreads, 1) kda_bwd_pass_tc_kernel(ChunkBwdArgs ca) {
  constexpr int DK = 128, DV = 128, NSL = DV / 32;
  using SM = PassTcSmem;
  using R = bwdc::Rec<DK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, half = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const BackwardArgs& ba = ca.b;
  const PrefillArgs& a = ba.f;
  const int sl = blockIdx.x % NSL, nh = blockIdx.x / NSL;
  const int n = nh / a.H, h = nh - n * a.H, col0 = 32 * sl;
  int64_t bq, t0;
  int len;
  bwdc::seq_span(a, n, bq, t0, len);
  const int nc = bwdc::num_chunks(ca, n), f0 = bwdc::first_chunk(ca, n);
  auto recp = [&](int c) { return ca.rec + ((int64_t)(f0 + c) * a.H + h) * R::SIZE; };
  auto stp = [&](int c) { return ca.st + ((int64_t)(f0 + c) * a.H + h) * R::SSIZE; };
  auto chunk = [&](int k) { return REV ? nc - 1 - k : k; };
  volatile int* sFlag = reinterpret_cast<volatile int*>(smem + SM::FLAG);
  float* xch = reinterpret_cast<float*>(smem + SM::XCH);
  const uint32_t mrec = s0 + SM::MBAR, mu = mrec + 16, ms = mrec + 24, mdone = mrec + 32;
  const int64_t m0off = REV ? R::WY : R::W;  // [hi; lo] tile, then the K_end / -beta K+ halves
  const int64_t voff = REV ? R::VY : R::UB;  // slice-major [64][32] rows
  constexpr uint32_t kRecBytes = REV ? 65536u + 16384u : 65536u;

  if (warp == 0) tmem_alloc(s0 + SM::SLOT, kPassTmemCols);
  if (tid == 0) {
    mbar_init(mrec, 1);
    mbar_init(mrec + 8, 1);
    mbar_init(mu, 1);
    mbar_init(ms, 1);
    mbar_init(mdone, 1);
    *sFlag = 0;
    fence_mbar_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM::SLOT);
  const uint32_t tS = tmem, tU = tmem + 64;
  const int d = 32 * q4 + lane;          // state row
  const int ir = 32 * (q4 & 1) + lane;   // chunk row of warps with q4 < 2
  const int cv = 16 * half;              // this thread's first state column
  // the starting state: S_0 (forward) or the final-state gradient (reverse); zero if absent
  {
    const float* init = REV ? (ba.dsT ? ba.dsT + n * ba.dsT_sn + h * ba.dsT_sh : nullptr)
                            : (a.s0 ? a.s0 + n * a.s0_sn + h * a.s0_sh : nullptr);
    uint32_t r[16], z[16];
#pragma unroll
    for (int t = 0; t < 16; t += 4) {
      const float4 x = init ? ld4(init + (int64_t)d * DV + col0 + cv + t) : zero4();
      r[t] = __float_as_uint(x.x), r[t + 1] = __float_as_uint(x.y), r[t + 2] = __float_as_uint(x.z),
      r[t + 3] = __float_as_uint(x.w);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) z[t] = 0u;
    tmem_st16_async(tS + lane_base + cv, r);
    tmem_st16_async(tS + lane_base + 32 + cv, z);
    tmem_wait_st();
  }
  // per-chunk vectors, one chunk ahead
  float eg = 0.f, vrow[16], be = 0.f;
  auto fetch = [&](int c) {
    const float* rc = recp(c);
    eg = rc[R::EGC + d];
    if (q4 < 2) {
#pragma unroll
      for (int k = 0; k < 16; k += 4) {
        const float4 x = ld4(rc + voff + sl * (kC * 32) + ir * 32 + cv + k);
        vrow[k] = x.x, vrow[k + 1] = x.y, vrow[k + 2] = x.z, vrow[k + 3] = x.w;
      }
      if (REV) {
        const int tok = c * kC + ir;
        be = tok < len ? a.beta[bq * a.beta_sb + (t0 + tok) * a.beta_st + (int64_t)h * a.beta_sh] : 0.f;
      }
    }
  };
  auto issue = [&](int k) {  // thread 0: chunk k's tiles (and Z_q slice) into buffer k & 1
    const uint32_t mb = mrec + 8 * (k & 1);
    const float* rc = recp(chunk(k));
    mbar_arrive_expect_tx(mb, kRecBytes);
    bulk_g2s(s0 + (uint32_t)(k & 1) * SM::BUF, rc + m0off, 65536u, mb);
    if (REV) bulk_g2s(s0 + SM::ZQB + (uint32_t)(k & 1) * 16384u, rc + R::ZQ + sl * (DK * 32), 16384u, mb);
  };
  // operand descriptors; a k-step adds a constant (in 16-byte units) to the address field
  const uint64_t dW0 = desc_kmajor(s0, 128, 0), dW1 = desc_kmajor(s0 + SM::BUF, 128, 0);
  const uint64_t dM0 = desc_mnmajor(s0 + SM::M1, kC, 0), dM1 = desc_mnmajor(s0 + SM::BUF + SM::M1, kC, 0);
  const uint64_t dSB = desc_mnmajor(s0 + SM::SB, 128, 0), dUB = desc_mnmajor(s0 + SM::UB, kC, 0);
  int issued = 0;  // bulk copies issued (chunks 0 .. issued - 1)
  if (tid == 0 && nc > 0) {
    issue(0);
    issued = 1;
  }
  if (nc > 0) fetch(chunk(0));
  fence_before_sync();
  __syncthreads();
  for (int k = 0; k < nc; ++k) {
    const int c = chunk(k), b = k & 1;
    if (tid == 0 && k + 1 < nc) {  // buffer b ^ 1 last served chunk k - 1, whose products are done
      issue(k + 1);
      issued = k + 2;
    }
    const float eg_c = eg, be_c = be;
    float v_c[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) v_c[t] = vrow[t];
    if (k + 1 < nc) fetch(chunk(k + 1));
    float* st = stp(c);
    // (1) the state entering this step (both accumulator halves): its bf16 halves (B of
    //     D_U), then decayed (plus Z_q) in place, the second half cleared
    float sv[16];
    {
      uint32_t ra[16], rb[16];
      tmem_ld16_async(tS + lane_base + cv, ra);
      tmem_ld16_async(tS + lane_base + 32 + cv, rb);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < 16; ++t) sv[t] = __uint_as_float(ra[t]) + __uint_as_float(rb[t]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = sv[8 * cc + e];
        store_split8(s0 + SM::SB + sw128(d, cv + 8 * cc, 128), s0 + SM::SB + sw128(d, 32 + cv + 8 * cc, 128), 0u, y);
      }
    }
    fence_async_smem();
    if (!mbar_wait(mrec + 8 * b, (uint32_t)((k >> 1) & 1))) *sFlag = 1;
    {
      float zq[16];
      if (REV) {  // Z_q row d, 16-byte chunks rotated by d
        const float* zr = reinterpret_cast<const float*>(smem + SM::ZQB + b * 16384) + d * 32;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 x = ld4(zr + 4 * ((4 * half + j + d) & 7));
          zq[4 * j] = x.x, zq[4 * j + 1] = x.y, zq[4 * j + 2] = x.z, zq[4 * j + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) zq[t] = 0.f;
      }
      uint32_t r[16], z[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        r[t] = __float_as_uint(eg_c * sv[t] + zq[t]);
        z[t] = 0u;
      }
      tmem_st16_async(tS + lane_base + cv, r);
      tmem_st16_async(tS + lane_base + 32 + cv, z);
      tmem_wait_st();
    }
    fence_before_sync();
    __syncthreads();
    if (*sFlag) goto fail;
    if (tid == 0) {
      fence_after_sync();
      const uint32_t idu = idesc_bf16(128, 64, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tU, (b ? dW1 : dW0) + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), dSB + (uint64_t)(ks * 128),
                 idu, ks > 0 ? 1u : 0u);
      mma_commit(mu);
    }
    {  // the state record, while D_U runs
      float* dst = st + (REV ? R::X : R::S) + (int64_t)d * DV + col0 + cv;
#pragma unroll
      for (int t = 0; t < 16; t += 4) st4(dst + t, make_float4(sv[t], sv[t + 1], sv[t + 2], sv[t + 3]));
    }
    if (!mbar_wait(mu, (uint32_t)(k & 1))) *sFlag = 1;
    fence_after_sync();
    // (2) U (or dY) rows: the high-half rows add the low-half rows through shared memory
    float y[16];
    {
      uint32_t ra[16], rb[16];
      tmem_ld16_async(tU + lane_base + cv, ra);
      tmem_ld16_async(tU + lane_base + 32 + cv, rb);
      tmem_wait_ld();
      float p[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) p[t] = __uint_as_float(ra[t]) + __uint_as_float(rb[t]);
      if (q4 >= 2)
#pragma unroll
        for (int t = 0; t < 16; ++t) xch[ir * SM::PX + cv + t] = p[t];
      __syncthreads();
      if (*sFlag) goto fail;
      if (q4 < 2) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float q = p[t] + xch[ir * SM::PX + cv + t];
          y[t] = REV ? v_c[t] + q : v_c[t] - q;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float z[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) z[e] = y[8 * cc + e];
          store_split8(s0 + SM::UB + sw128(ir, cv + 8 * cc, 64), s0 + SM::UB + sw128(ir, 32 + cv + 8 * cc, 64), 0u, z);
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      const uint32_t i64 = idesc_bf16(128, 64, true, true), i32 = idesc_bf16(128, 32, true, true);
      const uint64_t am = b ? dM1 : dM0;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tS, am + (uint64_t)(ks * 128), dUB + (uint64_t)(ks * 128), i64, 1u);          // K_hi [U_hi | U_lo]
        mma_bf16(tS, am + (uint64_t)(ks * 128 + 1024), dUB + (uint64_t)(ks * 128), i32, 1u);   // K_lo U_hi
      }
      mma_commit(ms);
    }
    if (q4 < 2) {  // the U (or dY) record and dv, while the state update runs
      float* dst = st + (REV ? R::DY : R::U) + (int64_t)ir * DV + col0 + cv;
#pragma unroll
      for (int t = 0; t < 16; t += 4) st4(dst + t, make_float4(y[t], y[t + 1], y[t + 2], y[t + 3]));
      const int tok = c * kC + ir;
      if (REV && tok < len) {
        float* dv = ba.dv.ptr + bq * ba.dv.sb + (t0 + tok) * ba.dv.st + (int64_t)h * ba.dv.sh + col0 + cv;
#pragma unroll
        for (int t = 0; t < 16; t += 4)
          st4(dv + t, make_float4(be_c * y[t], be_c * y[t + 1], be_c * y[t + 2], be_c * y[t + 3]));
      }
    }
    if (!mbar_wait(ms, (uint32_t)(k & 1))) *sFlag = 1;
    fence_after_sync();
    __syncthreads();
    if (*sFlag) goto fail;
  }
  // reverse: the initial-state gradient is the last X
  if (REV && ba.ds0) {
    uint32_t ra[16], rb[16];
    tmem_ld16_async(tS + lane_base + cv, ra);
    tmem_ld16_async(tS + lane_base + 32 + cv, rb);
    tmem_wait_ld();
    float* dst = ba.ds0 + n * ba.ds0_sn + h * ba.ds0_sh + (int64_t)d * DV + col0 + cv;
#pragma unroll
    for (int t = 0; t < 16; t += 4)
      st4(dst + t, make_float4(__uint_as_float(ra[t]) + __uint_as_float(rb[t]),
                               __uint_as_float(ra[t + 1]) + __uint_as_float(rb[t + 1]),
                               __uint_as_float(ra[t + 2]) + __uint_as_float(rb[t + 2]),
                               __uint_as_float(ra[t + 3]) + __uint_as_float(rb[t + 3])));
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kPassTmemCols);
  }
  return;

fail:
  // a wait gave up: report it, let what was issued finish (bounded), free the tensor memory
  if (tid == 0) {
    atomicOr(a.err, kErrTimeout);
    mma_commit(mdone);
    mbar_wait(mdone, 0);
    for (int k = (issued > 2 ? issued - 2 : 0); k < issued; ++k) mbar_wait(mrec + 8 * (k & 1), (uint32_t)((k >> 1) & 1));
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kPassTmemCols);
  }
}

}  // namespace

bool chunk_grad_tc_supported(const PrefillArgs& a) { return a.dk == 128 && a.dv == 128 && a.bf16; }

cudaError_t launch_chunk_grad_tc(const bwdc::ChunkBwdArgs& ca, cudaStream_t s) {
  const PrefillArgs& a = ca.b.f;
  if (!chunk_grad_tc_supported(a)) return cudaErrorInvalidValue;
  auto* k = kda_bwd_grad_tc_kernel<__nv_bfloat16>;
  constexpr int bytes = (int)GradTcSmem::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  launch_begin(s);
  k<<<dim3((unsigned)ca.total, (unsigned)a.H), kTcThreads, bytes, s>>>(ca);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

cudaError_t launch_chunk_pass_tc(const bwdc::ChunkBwdArgs& ca, bool reverse, cudaStream_t s) {
  const PrefillArgs& a = ca.b.f;
  if (!chunk_grad_tc_supported(a)) return cudaErrorInvalidValue;
  auto* k = reverse ? kda_bwd_pass_tc_kernel<true> : kda_bwd_pass_tc_kernel<false>;
  constexpr int bytes = (int)PassTcSmem::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((int64_t)a.N * a.H * (a.dv / 32));
  launch_begin(s);
  k<<<grid, kTcThreads, bytes, s>>>(ca);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

cudaError_t launch_chunk_prep_tc(const bwdc::ChunkBwdArgs& ca, cudaStream_t s) {
  const PrefillArgs& a = ca.b.f;
  if (!chunk_grad_tc_supported(a)) return cudaErrorInvalidValue;
  auto* k = kda_bwd_prep_tc_kernel<__nv_bfloat16>;
  constexpr int bytes = (int)PrepTcSmem::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  launch_begin(s);
  k<<<dim3((unsigned)ca.total, (unsigned)a.H), kTcThreads, bytes, s>>>(ca);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_end(s);
}

}  // namespace kda
