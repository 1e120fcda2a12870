// Internal interface between the C-ABI layer (kda_api.cu) and the kernel files.
// Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Device error word bits (or-ed by kernels, read by kda_get_device_error).
enum : int {
  kErrBadSeqlens = 1,  // cu_seqlens not starting at 0, decreasing or not ending at T
  kErrTimeout = 2,     // a bounded wait gave up
  kErrDomain = 4,      // (KDA_VALIDATE) an input outside its documented domain
};

// Strided view of a [B, T, H, D] (or [N, H, D]) activation; strides in elements.
struct Act {
  const void* ptr;
  int64_t sb, st, sh;  // batch, time, head strides (innermost stride is 1)
};

struct PrefillArgs {
  Act q, k, v, g;
  const float* beta;
  int64_t beta_sb, beta_st, beta_sh;
  const float* s0;  // nullable; [N, H, dk, dv] with strides s_sn, s_sh (inner contiguous)
  int64_t s0_sn, s0_sh;
  float* sT;  // nullable
  int64_t sT_sn, sT_sh;
  void* out;  // nullable for the recurrent kernel (no outputs)
  int64_t out_sb, out_st, out_sh;
  const int32_t* cu_seqlens;  // nullable
  // nullable (recurrent kernel only): per-sequence count of tokens whose state
  // update is kept; the final state is the state after that many tokens (clamped
  // to [0, length]) and is not written when the count is 0
  const int32_t* accepted;
  // gate: 0 = g holds the per-token log-decay (fp32); 1 = g holds decay logits z
  // in the q/k/v dtype and the log-decay is -5 sigmoid(gate_scale[h] z)
  int gate;
  const float* gate_scale;  // [H] (gate == 1)
  // nullable: state checkpoints [N * ck_count, H, dk, dv] fp32 (inner block
  // contiguous); checkpoint j of sequence n (row n * ck_count + j) is the state
  // after (j + 1) * ck_tokens tokens of that sequence, written when j < ck_count
  float* ckpt;
  int64_t ck_sr, ck_sh;  // row (n * ck_count + j) and head strides
  int ck_count, ck_tokens;
  int B, T, H, N, dk, dv;
  int bf16;  // 1: q/k/v/out are bf16, 0: fp32
  float scale;
  int* err;  // device error word
  // tests of the timeout path only (kda_test_stall_next_prefill): the chunked
  // serial kernel issues no record copies, so its bounded waits give up
  int test_stall;
};

struct DecodeArgs {
  float* state;
  int64_t s_sn, s_sh;
  Act q, k, v, g;  // sb = request stride, sh = head stride (st unused)
  const float* beta;
  int64_t beta_sn, beta_sh;
  void* out;
  int64_t out_sn, out_sh;
  int N, H, dk, dv;
  int bf16;
  float scale;
};

// Decode step with the layer's front and back ends (kda_recurrent.cu):
// short causal convolutions of q, k, v over cached raw inputs, SiLU, L2 norm of
// q and k, the step, then head RMSNorm and a sigmoid output gate.
struct FusedDecodeArgs {
  DecodeArgs d;  // q, k, v hold the raw (pre-convolution) inputs; out gets the gated output
  // conv caches [N, 3, H, dim] in the q/k/v dtype: the last three raw inputs, oldest first
  void* cq;
  void* ck;
  void* cv;
  int64_t cq_sn, cq_ss, cq_sh, ck_sn, ck_ss, ck_sh, cv_sn, cv_ss, cv_sh;
  const float* wq;  // conv weights [H, dim, 4] fp32, contiguous; [..., 3] multiplies the current input
  const float* wk;
  const float* wv;
  Act gate;                 // output-gate logits [N, H, dv] (sb = request stride, sh = head stride)
  const float* norm_w;      // [dv] fp32 or null
  float eps;                // RMSNorm epsilon
};

// Backward of the KDA core (kda_recurrent.cu): gradients with respect to q, k, v,
// g, beta and the initial state, all fp32.
struct GradAct {
  float* ptr;
  int64_t sb, st, sh;
};
struct BackwardArgs {
  PrefillArgs f;   // forward inputs (out, sT, err unused)
  Act dout;        // gradient of out, q's dtype
  const float* dsT;  // gradient of the final state [N, H, dk, dv] or null
  int64_t dsT_sn, dsT_sh;
  GradAct dq, dk, dv, dg;  // [B, T, H, d] fp32
  float* dbeta;            // [B, T, H] fp32
  int64_t db_sb, db_st, db_sh;
  float* ds0;              // [N, H, dk, dv] fp32 or null
  int64_t ds0_sn, ds0_sh;
  float* ck;   // workspace: states every kBwdBlock tokens, [N * H][nblk][dk][dv]
  float* scr;  // workspace: the states entering each token of one block, [N * H][kBwdBlock][dk][dv]
  float* part; // workspace when d_v is split four ways: the row sums of slices 2-3,
               // [B * T * H][4][dk] (dq, dk, dg, dbeta at [3][0]); else null
  int nblk;    // ceil(T / kBwdBlock)
};
constexpr int kBwdBlock = 32;
// value-column slices per (sequence, head) of the backward kernel (1, 2 or 4)
int backward_value_slices(int N, int H, int dv);
// rows = B * T (the token rows of the inputs)
size_t backward_workspace_bytes(int N, int H, int T, int64_t rows, int dk, int dv);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);

// SIMT kernels (kda_recurrent.cu)
// ws: decode_fused_workspace_bytes(N, H, dk, dv) bytes of device scratch
cudaError_t launch_decode_fused(const FusedDecodeArgs& a, void* ws, cudaStream_t s);
size_t decode_fused_workspace_bytes(int N, int H, int dk, int dv);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_recurrent_prefill(const PrefillArgs& a, cudaStream_t s);
// cu_seqlens validation: sets kErrBadSeqlens in *err when the offsets are invalid.
cudaError_t launch_check_seqlens(const int32_t* cu, int N, int T, int* err, cudaStream_t s);

// Tensor-core chunked prefill (kda_prefill_tc.cu); bf16 inputs only.  The
// workspace (device memory, chunk_prefill_workspace_bytes(a) bytes, 1024-byte
// aligned) holds the per-chunk records; it is only used by work enqueued on `s`.
size_t chunk_prefill_workspace_bytes(const PrefillArgs& a);
cudaError_t launch_chunk_prefill_tc(const PrefillArgs& a, void* workspace, cudaStream_t s);

// Size of the fixed device workspace behind kda_chunk_fwd_noalloc, and its
// device address on the current device (kda_noalloc.cu; looked up once per device).
constexpr size_t kNoallocWorkspaceBytes = size_t(64) << 20;
cudaError_t noalloc_workspace(void** ptr);

// Launch accounting (kda_api.cu): every kernel launch is bracketed by
// launch_begin (before) and launch_end (after its own launch check succeeded).
// launch_end returns the error of recording an armed event, if any.
void launch_begin(cudaStream_t s);
cudaError_t launch_end(cudaStream_t s);

// Input-domain checks (kda_validate.cu), enabled by KDA_VALIDATE in the environment:
// q, k, v finite; g in [-5, 0] (or, with the gate, finite logits and gate scales);
// beta in [0, 1].  Rows are (b, t, h) for b < B, t < T, h < H.
struct ValidateArgs {
  Act q, k, v, g;
  const float* beta;
  int64_t beta_sb, beta_st, beta_sh;
  const float* gate_scale;  // [H] or null
  int B, T, H, dk, dv;
  int bf16;  // q, k, v (and gate logits) are bf16
  int gate;  // g holds decay logits in q's dtype
  int* err;
};
bool validate_enabled();
cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s);

// SM count of the current device, cached per device (kda_prefill_tc.cu).
int sm_count();

// Stream-ordered scratch memory from a per-device pool (kda_api.cu).
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);

}  // namespace kda
