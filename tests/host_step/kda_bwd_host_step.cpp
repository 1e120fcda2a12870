// Steps the chunked-backward kernel bodies (kda_backward_chunk.cuh) on the host:
// every CUDA block runs as one std::thread per CUDA thread, with std::barrier as
// the block barrier and host vectors as shared memory (filled with NaN first, so a
// read before a write shows up in the results).  Test infrastructure only: built
// by tests/test_chunk_bwd_host_step.py, never by the library.
//
//   host_step_backward(...)  the four kernels of kda_chunk_bwd on host arrays
//                            (fp32 inputs, contiguous [B, T, H, d] layouts)
//   main()                   (with -DKB_HOST_STEP_MAIN) runs a fixed set of
//                            shapes on random inputs; built with AddressSanitizer
//                            it checks every shared and global access for bounds
#include <barrier>
#include <cmath>
#include <cstdio>
#include <thread>
#include <vector>

static thread_local std::barrier<>* kb_bar = nullptr;
#define KB_SYNC() kb_bar->arrive_and_wait()
#include "kda_backward_chunk.cuh"

using namespace kda;
using namespace kda::bwdc;

namespace {

template <class F>
void run_block(int nt, size_t smem_floats, F body) {
  std::vector<float> sm(smem_floats, std::nanf(""));
  std::barrier<> bar(nt);
  std::vector<std::thread> th;
  th.reserve(nt);
  for (int t = 0; t < nt; ++t)
    th.emplace_back([&, t] {
      kb_bar = &bar;
      body(sm.data(), t);
    });
  for (auto& x : th) x.join();
}

template <int DK, int DV>
void run_all(ChunkBwdArgs& ca) {
  const PrefillArgs& a = ca.b.f;
  for (int h = 0; h < a.H; ++h)
    for (int f = 0; f < ca.total; ++f)
      run_block(256, PrepSmem<DK, DV>::FLOATS, [&](float* sm, int t) { prep_body<DK, DV, float>(ca, sm, f, h, t); });
  const int np = a.N * a.H * (DV / kW);
  for (int b = 0; b < np; ++b)
    run_block(kPassThreads, PassSmem<DK>::FLOATS,
              [&](float* sm, int t) { pass_body<DK, DV, float, false>(ca, sm, b, t); });
  for (int b = 0; b < np; ++b)
    run_block(kPassThreads, PassSmem<DK>::FLOATS,
              [&](float* sm, int t) { pass_body<DK, DV, float, true>(ca, sm, b, t); });
  for (int h = 0; h < a.H; ++h)
    for (int f = 0; f < ca.total; ++f)
      run_block(256, GradSmem<DK, DV>::FLOATS, [&](float* sm, int t) { grad_body<DK, DV, float>(ca, sm, f, h, t); });
}

}  // namespace

// Gradients of the KDA core for fp32 inputs in contiguous layouts; s0, cu, dsT and
// ds0 may be null.  Returns 0, or 1 for an unsupported head-dim pair.
extern "C" int host_step_backward(int B, int T, int H, int dk, int dv, const float* q, const float* k,
                                  const float* v, const float* g, const float* beta, const float* s0,
                                  float scale, const int* cu, int N, const float* dout, const float* dsT,
                                  float* dq, float* dkk, float* dvv, float* dg, float* db, float* ds0) {
  ChunkBwdArgs ca{};
  BackwardArgs& ba = ca.b;
  PrefillArgs& a = ba.f;
  auto act = [&](const float* p, int d) {
    Act x;
    x.ptr = p;
    x.sb = (int64_t)T * H * d;
    x.st = (int64_t)H * d;
    x.sh = d;
    return x;
  };
  auto gact = [&](float* p, int d) {
    GradAct x;
    x.ptr = p;
    x.sb = (int64_t)T * H * d;
    x.st = (int64_t)H * d;
    x.sh = d;
    return x;
  };
  const int64_t state = (int64_t)dk * dv;
  a.q = act(q, dk);
  a.k = act(k, dk);
  a.v = act(v, dv);
  a.g = act(g, dk);
  a.beta = beta;
  a.beta_sb = (int64_t)T * H;
  a.beta_st = H;
  a.beta_sh = 1;
  a.s0 = s0;
  a.s0_sn = H * state;
  a.s0_sh = state;
  a.cu_seqlens = cu;
  a.B = B;
  a.T = T;
  a.H = H;
  a.N = N;
  a.dk = dk;
  a.dv = dv;
  a.scale = scale;
  ba.dout = act(dout, dv);
  ba.dsT = dsT;
  ba.dsT_sn = H * state;
  ba.dsT_sh = state;
  ba.dq = gact(dq, dk);
  ba.dk = gact(dkk, dk);
  ba.dv = gact(dvv, dv);
  ba.dg = gact(dg, dk);
  ba.dbeta = db;
  ba.db_sb = (int64_t)T * H;
  ba.db_st = H;
  ba.db_sh = 1;
  ba.ds0 = ds0;
  ba.ds0_sn = H * state;
  ba.ds0_sh = state;
  const int nck = (T + kC - 1) / kC;
  ca.nck = nck;
  ca.total = cu ? nck + N : nck * N;
  std::vector<int> off;
  if (cu) {  // the chunk offsets the library's offsets kernel computes
    off.resize(N + 1);
    int run = 0;
    for (int n = 0; n < N; ++n) {
      off[n] = run;
      int64_t b, t0;
      int len;
      seq_span(a, n, b, t0, len);
      run += (len + kC - 1) / kC;
    }
    off[N] = run;
    ca.off = off.data();
  }
  const size_t recf = (size_t)4 * kC * dk + 2 * kC * dv + dk + (size_t)dk * dv + kC * kC;
  const size_t stf = (size_t)2 * dk * dv + 2 * kC * dv;
  std::vector<float> rec((size_t)ca.total * H * recf, std::nanf("")), st((size_t)ca.total * H * stf, std::nanf(""));
  ca.rec = rec.data();
  ca.st = st.data();
  if (dk == 64 && dv == 64) run_all<64, 64>(ca);
  else if (dk == 64 && dv == 128) run_all<64, 128>(ca);
  else if (dk == 128 && dv == 64) run_all<128, 64>(ca);
  else if (dk == 128 && dv == 128) run_all<128, 128>(ca);
  else return 1;
  return 0;
}

#ifdef KB_HOST_STEP_MAIN
#include <random>
int main() {
  struct Case {
    int B, T, H, dk, dv;
    std::vector<int> lens;
    bool s0, dst;
  };
  const std::vector<Case> cases = {
      {1, 1, 1, 64, 64, {}, true, true},          {2, 64, 2, 64, 64, {}, false, false},
      {1, 65, 1, 128, 128, {}, true, true},       {1, 150, 2, 64, 128, {}, true, true},
      {1, 130, 1, 128, 64, {}, true, false},      {1, 181, 2, 64, 64, {0, 40, 1, 70, 0, 70}, true, true},
      {1, 129, 1, 128, 128, {0, 129}, false, true}, {1, 0, 1, 64, 64, {0, 0}, true, true}};
  std::mt19937 rng(1);
  std::normal_distribution<float> nd;
  int bad = 0;
  for (const auto& c : cases) {
    const int N = c.lens.empty() ? c.B : (int)c.lens.size();
    auto vec = [&](size_t n) {
      std::vector<float> x(n);
      for (auto& y : x) y = 0.3f * nd(rng);
      return x;
    };
    const size_t rk = (size_t)c.B * c.T * c.H * c.dk, rv = (size_t)c.B * c.T * c.H * c.dv, rb = (size_t)c.B * c.T * c.H;
    const size_t ns = (size_t)N * c.H * c.dk * c.dv;
    auto q = vec(rk), k = vec(rk), v = vec(rv), g = vec(rk), beta = vec(rb), dout = vec(rv), s0 = vec(ns), dst = vec(ns);
    for (auto& x : g) x = -std::fabs(x);
    std::vector<int> cu;
    if (!c.lens.empty()) {
      cu.push_back(0);
      for (int l : c.lens) cu.push_back(cu.back() + l);
    }
    std::vector<float> dq(rk), dk(rk), dv(rv), dg(rk), db(rb), ds0(ns);
    const int rc = host_step_backward(c.B, c.T, c.H, c.dk, c.dv, q.data(), k.data(), v.data(), g.data(), beta.data(),
                                      c.s0 ? s0.data() : nullptr, 0.5f, cu.empty() ? nullptr : cu.data(), N,
                                      dout.data(), c.dst ? dst.data() : nullptr, dq.data(), dk.data(), dv.data(),
                                      dg.data(), db.data(), ds0.data());
    bool finite = true;
    for (const auto* vv : {&dq, &dk, &dv, &dg, &db, &ds0})
      for (float x : *vv) finite = finite && std::isfinite(x);
    std::printf("B%d T%d H%d %dx%d rc=%d finite=%d\n", c.B, c.T, c.H, c.dk, c.dv, rc, (int)finite);
    bad += rc != 0 || !finite;
  }
  return bad;
}
#endif
