// KDA oracle: plain fp64 token-by-token recurrence on the CPU.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load or call this
// file; only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg
// use it.  It shares no code, header or constant with the CUDA library.
//
// What it computes (for every independent problem = one sequence of one head):
//   S <- S0 (or 0)
//   for t in order:
//     S <- Diag(exp(g_t)) S                       (1) decay
//     S <- S - beta_t k_t (k_t^T S)                (2) rank-1 correction
//     S <- S + beta_t k_t v_t^T                    (3) write
//     o_t <- scale * S^T q_t                       read-out after the update
//   S_T <- S
// This is the KDA state update S_t = (I - beta k k^T) Diag(alpha_t) S_{t-1}
// + beta k v^T with alpha_t = exp(g_t): "Kimi K3 核心算子拆解" (devpress.csdn.net)
// §2.2 and its three-step decomposition §2.3; the read-out o_t = S_t^T q_t
// after the update is "Kimi K3 技术报告解读" (marsggbo.github.io) §3.2-§3.3.
// The order of (2) then (3) is the pages' three-step order; it makes the row of
// S along a unit key equal v_t exactly.
//
// Layout: problem p owns the rows [row_start[p], row_start[p] + row_count[p]) of
// the row-major arrays q, k, g ([rows][dk]), v, out ([rows][dv]) and beta
// ([rows]); problems must not share rows.  S0 (nullable) and S_out are
// [P][dk][dv].  Problems run in parallel (OpenMP).
#include <cmath>
#include <cstdint>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

void run_problem(int64_t t0, int64_t t1, int dk, int dv, const double* q, const double* k,
                 const double* v, const double* g, const double* beta, const double* s0,
                 double scale, double* out, double* s_out) {
  std::vector<double> S(static_cast<size_t>(dk) * dv, 0.0);
  std::vector<double> kS(dv), alpha(dk);
  if (s0)
    for (size_t i = 0; i < S.size(); ++i) S[i] = s0[i];
  for (int64_t t = t0; t < t1; ++t) {
    const double* qt = q + t * dk;
    const double* kt = k + t * dk;
    const double* vt = v + t * dv;
    const double* gt = g + t * dk;
    const double bt = beta[t];
    for (int i = 0; i < dk; ++i) alpha[i] = std::exp(gt[i]);
    // (1) decay each key-channel row of S
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[static_cast<size_t>(i) * dv + j] *= alpha[i];
    // (2) kS = k^T S (decayed);  S -= beta k kS^T
    for (int j = 0; j < dv; ++j) kS[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) kS[j] += kt[i] * S[static_cast<size_t>(i) * dv + j];
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[static_cast<size_t>(i) * dv + j] -= bt * kt[i] * kS[j];
    // (3) S += beta k v^T
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[static_cast<size_t>(i) * dv + j] += bt * kt[i] * vt[j];
    // read-out o_t = scale * S^T q_t
    double* ot = out + t * dv;
    for (int j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) ot[j] += qt[i] * S[static_cast<size_t>(i) * dv + j];
    for (int j = 0; j < dv; ++j) ot[j] *= scale;
  }
  for (size_t i = 0; i < S.size(); ++i) s_out[i] = S[i];
}

}  // namespace

extern "C" {

// Number of threads a parallel region of this library would use (nthreads <= 0
// means the OpenMP default).
int kda_oracle_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

// Runs P independent problems.  Returns the number of threads used, or a
// negative value on invalid arguments.
int kda_oracle_run(int64_t P, const int64_t* row_start, const int64_t* row_count, int dk,
                   int dv, const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* s0, double scale, double* out,
                   double* s_out, int nthreads) {
  if (P < 0 || dk <= 0 || dv <= 0 || !row_start || !row_count || !s_out) return -1;
  for (int64_t p = 0; p < P; ++p)
    if (row_start[p] < 0 || row_count[p] < 0) return -2;
  const int nt = kda_oracle_threads(nthreads);
  const size_t st = static_cast<size_t>(dk) * dv;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
  for (int64_t p = 0; p < P; ++p)
    run_problem(row_start[p], row_start[p] + row_count[p], dk, dv, q, k, v, g, beta,
                s0 ? s0 + p * st : nullptr, scale, out, s_out + p * st);
  return nt;
}

}  // extern "C"
