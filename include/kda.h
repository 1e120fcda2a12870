/*
 * libkda - Kimi Delta Attention (KDA) core for NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence and head, state S in R^{d_k x d_v}, fp32):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t                      (read-out after the update)
 *
 * Sources: "Kimi K3 核心算子拆解" (devpress.csdn.net) §2.2 (state update) and
 * §2.3 (decay / rank-1 correction / write); "Kimi K3 技术报告解读"
 * (marsggbo.github.io) §3.2 (read-out S_t^T q_t) and §3.5 (log-decay g bounded
 * in (-5, 0)); chunked prefill: "尝试对Kimi KDA的数学推导&算子实现分析"
 * (hjcheng0602.cn/blog/kdd) eqs. (9)-(66).
 *
 * Conventions shared by every entry point
 *  - Tensors are passed as kda_tensor descriptors: a DEVICE pointer, a dtype,
 *    a rank and per-dimension sizes and strides counted in ELEMENTS.  The
 *    caller owns every buffer; the library keeps no pointer after a call
 *    returns.  The innermost dimension must be contiguous (stride 1) and every
 *    data pointer and every outer stride (in bytes) a multiple of 16.
 *  - g is the PER-TOKEN log-decay (alpha = exp(g)); its documented domain is
 *    [-5, 0] and beta's is [0, 1].  Outside it results follow the definition
 *    above but may lose precision.  q and k are expected L2-normalised by the
 *    caller (the KDA layer does this before the core); the library does not
 *    normalise them.
 *  - Head dimensions d_k, d_v are each 64 or 128.
 *  - q, k, v (and out) share one dtype: KDA_DTYPE_BF16 or KDA_DTYPE_F32.
 *    g, beta and the states are always KDA_DTYPE_F32.  out has q's dtype,
 *    rounded to nearest even from fp32 accumulators.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream).  KDA_OK means "validated and enqueued".
 *  - Errors the host can detect return KDA_ERR_INVALID_ARG or
 *    KDA_ERR_UNSUPPORTED before anything is launched and set a thread-local
 *    message (kda_last_error_message).  A failed launch returns KDA_ERR_CUDA.
 *    Problems only the device can see (cu_seqlens not non-decreasing, not
 *    starting at 0 or not ending at T) are recorded in a per-device error word
 *    read by kda_get_device_error; outputs are then unspecified.  NaN inputs
 *    propagate; nothing traps.
 *  - Input-domain checks (optional): with KDA_VALIDATE set to a non-empty value
 *    other than "0" in the environment (read at every call), every compute
 *    entry point first enqueues one extra kernel that reads q, k, v, g (or the
 *    gate logits) and beta once and records KDA_ERR_DOMAIN in the device error
 *    word if a value is not finite, a g is outside [-5, 0] or a beta outside
 *    [0, 1] (the bounded decay of "Kimi K3 技术报告解读" (marsggbo.github.io)
 *    §3.5, which the chunked kernels rely on for exponent safety).  The check
 *    changes no result; it costs one extra read of the inputs.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* a descriptor, shape, dtype, stride, alias or value is invalid */
  KDA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (e.g. d_k = 96) */
  KDA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  KDA_ERR_DEVICE = 4,      /* the device reported bad cu_seqlens (kda_get_device_error) */
  KDA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (kda_get_device_error) */
  KDA_ERR_DOMAIN = 6       /* KDA_VALIDATE found an input outside its domain (kda_get_device_error) */
} kda_status;

typedef enum kda_dtype {
  KDA_DTYPE_F32 = 0,
  KDA_DTYPE_BF16 = 1,
  KDA_DTYPE_I32 = 2
} kda_dtype;

typedef struct kda_tensor {
  void* data;        /* device pointer */
  int32_t dtype;     /* kda_dtype */
  int32_t ndim;      /* 1..4 */
  int64_t shape[4];  /* sizes of the first ndim dimensions */
  int64_t stride[4]; /* strides in elements; stride[ndim-1] must be 1 */
} kda_tensor;

/*
 * kda_chunk_fwd - chunkwise-parallel prefill (forward) of the KDA core.
 *
 * Defined by the recurrence above, computed chunk by chunk as in
 * "尝试对Kimi KDA的数学推导&算子实现分析" (hjcheng0602.cn/blog/kdd): in-chunk
 * cumulative log-decay (eq. 9), strictly lower-triangular A / L (eqs. 22, 51),
 * triangular solve for U (eq. 52), output (eq. 63), state passed between
 * chunks (eqs. 64-66).
 *
 *   q, k          [B, T, H, d_k]  bf16 or f32
 *   v             [B, T, H, d_v]  same dtype as q
 *   g             [B, T, H, d_k]  f32, per-token log-decay
 *   beta          [B, T, H]       f32
 *   initial_state [N, H, d_k, d_v] f32, inner [d_k, d_v] contiguous; NULL = zeros
 *   scale         finite float multiplying the read-out (usually 1/sqrt(d_k))
 *   cu_seqlens    NULL: N = B and every batch row is one sequence of T tokens.
 *                 Otherwise [N+1] int32 on the device, B must be 1, and
 *                 sequence n is tokens [cu_seqlens[n], cu_seqlens[n+1]) of the
 *                 packed batch; values must start at 0, never decrease and end
 *                 at T (checked on the device).  No state crosses a boundary:
 *                 each sequence's results equal those of the sequence alone.
 *   out           [B, T, H, d_v]  q's dtype; written for every token
 *   final_state   [N, H, d_k, d_v] f32 or NULL; may be the same tensor as
 *                 initial_state (in place) but must not partly overlap it.
 *   stream        cudaStream_t as void*
 *
 * out must not overlap any input.  Empty sequences are allowed (their final
 * state is their initial state).  fp32 inputs run the recurrence itself in
 * fp32 (error well under 1e-4); bf16 inputs run the chunked tensor-core path
 * with fp32 accumulation and an fp32 state.
 */
kda_status kda_chunk_fwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta,
                         const kda_tensor* initial_state, float scale,
                         const kda_tensor* cu_seqlens, kda_tensor* out,
                         kda_tensor* final_state, void* stream);

/*
 * kda_fused_recurrent_fwd - the same operation and contract as kda_chunk_fwd,
 * computed by the recurrence itself with each (sequence, head) state held on
 * chip in fp32, four tokens per pass over the state (the single step unrolled
 * over four tokens: the same values up to fp32 rounding) ("把注意力换成一块「会遗忘的内存」" (jokeuncle.github.io), section on
 * the layer's two execution paths: short sequences use the fused recurrent
 * kernel).  Meant for short sequences and as an independent device-side
 * cross-check of the chunked path; kda_chunk_fwd uses it for fp32 inputs.
 */
kda_status kda_fused_recurrent_fwd(const kda_tensor* q, const kda_tensor* k,
                                   const kda_tensor* v, const kda_tensor* g,
                                   const kda_tensor* beta, const kda_tensor* initial_state,
                                   float scale, const kda_tensor* cu_seqlens, kda_tensor* out,
                                   kda_tensor* final_state, void* stream);

/*
 * kda_chunk_fwd_noalloc - kda_chunk_fwd for callers that must not allocate.
 *
 * The pages have no counterpart for this entry point; it exists for callers
 * that cannot call cudaMalloc or any allocating routine during a call: hosts
 * whose device memory is fully pre-sized and owned by their own allocator, and
 * code paths where allocation is not permitted.  It computes exactly what
 * kda_chunk_fwd computes, with the same arguments, layouts and errors, but
 * keeps the bf16 path's per-chunk records in a fixed 64 MiB device array
 * built into the library instead of pool memory (fp32 inputs need no scratch).
 *
 *  - The array is allocated on every device that loads the library and stays
 *    there until the process exits.
 *  - Requests whose records would not fit return KDA_ERR_UNSUPPORTED before
 *    anything is launched.  The records take 66560 bytes per (chunk, head)
 *    at d_k = 128 and 41984 at d_k = 64, over B * ceil(T / 64) chunks (with
 *    cu_seqlens: ceil(T / 64) + N, plus a small offset table), so at most
 *    1008 (chunk, head) pairs at d_k = 128, e.g. B=1, H=15, T=4096.  A
 *    sequence longer than 1152 chunks (73728 tokens) also needs, per head and
 *    per 128-chunk segment after its first, d_k * (2 d_v + d_k) * 4 bytes
 *    (192 KiB at d_k = d_v = 128) of segment states; with cu_seqlens that room
 *    is set aside for every 128 chunks of the call.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls share the one array.  Nothing in it has to start zeroed (every
 *    byte a call reads is written earlier in the same call), but two calls
 *    that run at the same time on the GPU, on any streams, overwrite each
 *    other's records: order them, e.g. on one stream.
 */
kda_status kda_chunk_fwd_noalloc(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                 const kda_tensor* g, const kda_tensor* beta,
                                 const kda_tensor* initial_state, float scale,
                                 const kda_tensor* cu_seqlens, kda_tensor* out,
                                 kda_tensor* final_state, void* stream);

/*
 * kda_recurrent_step - one decode token per request, state updated in place.
 *
 * The single-step recurrence in the three steps of "Kimi K3 核心算子拆解"
 * §2.3 (decay, rank-1 correction, write), fused so each state element is read
 * once and written once.
 *
 *   state  [N, H, d_k, d_v] f32, inner [d_k, d_v] contiguous; read and
 *          overwritten with S_t
 *   q, k   [N, H, d_k]  bf16 or f32
 *   v      [N, H, d_v]  same dtype as q
 *   g      [N, H, d_k]  f32
 *   beta   [N, H]       f32
 *   out    [N, H, d_v]  q's dtype
 *
 * out must not overlap state or any input.  With beta = 1 and k a unit basis
 * vector e_i the new row i of the state equals v exactly.
 */
kda_status kda_recurrent_step(kda_tensor* state, const kda_tensor* q, const kda_tensor* k,
                              const kda_tensor* v, const kda_tensor* g,
                              const kda_tensor* beta, float scale, kda_tensor* out,
                              void* stream);

/*
 * kda_chunk_fwd_checkpointed - kda_chunk_fwd that also writes the state at
 * regular token boundaries of every sequence (prefix-cache checkpoints).
 *
 * "Kimi K3 技术报告解读" (marsggbo.github.io) §9: prefixes are matched on
 * 512-token hash blocks and the KDA state is checkpointed only at sparse block
 * boundaries; a hit restores the nearest checkpoint and continues the prefill
 * from there.  Checkpoint j of sequence n is the state after the first
 * (j + 1) * checkpoint_tokens tokens of that sequence, exactly the state the
 * chunked recurrence holds there, so a prefill resumed from it (initial_state =
 * the checkpoint, inputs = the rest of the sequence) continues the original
 * run; without the segment split (sequences of at most 73728 tokens) the resumed
 * outputs and final state are bit-identical.
 *
 *   checkpoint_tokens  positive multiple of 64 (the chunk length)
 *   checkpoints        [N * C, H, d_k, d_v] f32, inner [d_k, d_v] contiguous:
 *                      row n * C + j holds checkpoint j of sequence n, for
 *                      j < min(C, length_n / checkpoint_tokens); other rows
 *                      are left as they are
 *   all other arguments, shapes, errors and guarantees as for kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_checkpointed(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                      const kda_tensor* g, const kda_tensor* beta,
                                      const kda_tensor* initial_state, float scale,
                                      const kda_tensor* cu_seqlens, int64_t checkpoint_tokens,
                                      kda_tensor* checkpoints, kda_tensor* out, kda_tensor* final_state,
                                      void* stream);

/*
 * kda_chunk_fwd_gated - kda_chunk_fwd with the log-decay formed in the kernel
 * from decay logits: g = -5 * sigmoid(gate_scale[h] * gate).
 *
 * "Kimi K3 技术报告解读" (marsggbo.github.io) §3.5 replaces the negative
 * softplus decay map by a scaled sigmoid of the decay logit z with a learnable
 * per-head scale A_h, so that every step keeps alpha > e^-5; the formula itself
 * is not legible in the page text, and this call takes the reading that keeps
 * that bound for any A_h: g = -5 sigmoid(A_h z).  "Kimi K3 四个核心模块的公式与
 * 真实张量流" (gentlecold.top) §1.5 names the fused-gate chunked kernel.  The
 * logits travel in the input dtype (bf16: 2 bytes per channel instead of 4).
 *
 *   gate        [B, T, H, d_k]  same dtype as q: decay logits z
 *   gate_scale  [H] f32 on the device: A_h
 *   all other arguments, shapes, errors and guarantees as for kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_gated(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                               const kda_tensor* gate, const kda_tensor* gate_scale,
                               const kda_tensor* beta, const kda_tensor* initial_state, float scale,
                               const kda_tensor* cu_seqlens, kda_tensor* out,
                               kda_tensor* final_state, void* stream);

/*
 * kda_backward - gradients of the KDA core: given the gradient d_out of the
 * outputs (and d_final_state of the final state, or NULL) of the forward that
 * kda_chunk_fwd computes from q, k, v, g, beta, initial_state, scale and
 * cu_seqlens, writes the gradients with respect to all of those inputs.
 *
 * The pages give the forward only ("尝试对Kimi KDA的数学推导&算子实现分析"
 * (hjcheng0602.cn/blog/kdd), the recurrence of "Kimi K3 核心算子拆解"
 * (devpress.csdn.net) §2.3); this is its exact reverse-mode derivative, run
 * token by token in reverse per (sequence, head) with the states recomputed from
 * checkpoints every 32 tokens.
 *
 *   q, k, v, g, beta, initial_state, scale, cu_seqlens  as for kda_chunk_fwd
 *   d_out            [B, T, H, d_v] in q's dtype
 *   d_final_state    [N, H, d_k, d_v] f32, or NULL (zero)
 *   dq, dk, dg       [B, T, H, d_k] f32;  dv [B, T, H, d_v] f32;  dbeta [B, T, H] f32
 *   d_initial_state  [N, H, d_k, d_v] f32, or NULL (not written)
 *
 * Scratch comes from the stream-ordered pool: N * H * (ceil(T / 32) + 32) *
 * d_k * d_v * 4 bytes, plus B * T * H * 4 * d_k * 4 bytes when d_v = 128 is
 * split over four 32-column CTAs per (sequence, head) (few sequence-heads).  The
 * result does not depend on the order in which those CTAs finish.  Errors as
 * for kda_chunk_fwd; no gradient may overlap an input or another gradient.
 */
kda_status kda_backward(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                        const kda_tensor* g, const kda_tensor* beta, const kda_tensor* initial_state,
                        float scale, const kda_tensor* cu_seqlens, const kda_tensor* d_out,
                        const kda_tensor* d_final_state, kda_tensor* dq, kda_tensor* dk, kda_tensor* dv,
                        kda_tensor* dg, kda_tensor* dbeta, kda_tensor* d_initial_state, void* stream);

/*
 * kda_chunk_bwd - the same gradients as kda_backward (same arguments, layouts
 * and errors), computed by the chunked form instead of the token loop.
 *
 * Per chunk of 64 tokens it differentiates the chunked equations of
 * "尝试对Kimi KDA的数学推导&算子实现分析" (hjcheng0602.cn/blog/kdd) eqs. (9),
 * (15)-(16), (36), (51)-(52), (63)-(66): a chunk-parallel kernel forms each
 * chunk's state-independent matrices, two sequential kernels carry the state
 * forward and its gradient backward through the chunks (per sequence, head and
 * 32 value columns; the reverse one writes dv), and a chunk-parallel kernel
 * forms dq, dk, dg and dbeta.  Like kda_chunk_fwd it relies on g in [-5, 0]
 * (cumulative decays inside a 16-token sub-block above -80; outside that range
 * use kda_backward).  The result is deterministic (no atomics).
 *
 * Scratch comes from the stream-ordered pool: per (chunk, head)
 * (4*64*d_k + 2*64*d_v + d_k + d_k*d_v + 64*64 + 2*d_k*d_v + 2*64*d_v) * 4 bytes,
 * about 475 KB at d_k = d_v = 128, over N * ceil(T / 64) chunks (ceil(T / 64) + N
 * with cu_seqlens).  A chunk count above 2^31 - 1 returns KDA_ERR_UNSUPPORTED
 * before any launch; otherwise errors as for kda_backward.
 */
kda_status kda_chunk_bwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta, const kda_tensor* initial_state,
                         float scale, const kda_tensor* cu_seqlens, const kda_tensor* d_out,
                         const kda_tensor* d_final_state, kda_tensor* dq, kda_tensor* dk, kda_tensor* dv,
                         kda_tensor* dg, kda_tensor* dbeta, kda_tensor* d_initial_state, void* stream);

/*
 * kda_decode_step_fused - one decode token per (request, head) with the KDA
 * layer's front and back ends fused around kda_recurrent_step.
 *
 * Front ("Kimi K3 四个核心模块的公式与真实张量流" (gentlecold.top) §1.2; "Kimi K3
 * 核心算子拆解" (devpress.csdn.net) §2.6): each of q, k, v passes a causal
 * depthwise convolution of width 4 over its three cached raw inputs and the new
 * one, then SiLU; q and k are L2-normalised (x / max(||x||, 1e-6)).  The caches
 * then drop their oldest input and take the new raw one.  Core: the decode step
 * on the processed q, k, v.  Back ("把注意力换成一块「会遗忘的内存」"
 * (jokeuncle.github.io), the sigmoid output gate of the layer's norm; devpress
 * §2.5): out = o / sqrt(mean(o^2) + eps) * norm_weight * sigmoid(out_gate), o the
 * step's read-out (scale * S^T q) over the head's d_v values.
 *
 *   state            [N, H, d_k, d_v] f32, inner block contiguous; in/out
 *   conv_q, conv_k   [N, 3, H, d_k] in q's dtype; conv_v [N, 3, H, d_v]: the last
 *                    three raw inputs, oldest first; in/out.  Pointer and strides
 *                    aligned to two elements (channels move in pairs)
 *   q, k             [N, H, d_k] raw (pre-convolution) inputs, bf16 or f32
 *   v                [N, H, d_v] raw, q's dtype
 *   w_q, w_k         [H, d_k, 4] f32 contiguous; w_v [H, d_v, 4]: convolution
 *                    weights, [..., 3] multiplying the new input
 *   g                [N, H, d_k] f32 log-decay; beta [N, H] f32
 *   out_gate         [N, H, d_v] q's dtype: output-gate logits
 *   norm_weight      [d_v] f32, or NULL (all ones)
 *   scale, eps       finite; eps >= 0
 *   out              [N, H, d_v] q's dtype
 *
 * Three kernels on `stream`: the front end writes the processed q, k, v in fp32
 * to scratch from the library's stream-ordered pool (N * H * (2 d_k + 2 d_v) * 4
 * bytes, released on the stream), the decode step reads them, and the back end
 * finishes the output.
 *
 * Errors as for kda_recurrent_step; no output may overlap another tensor.
 */
kda_status kda_decode_step_fused(kda_tensor* state, kda_tensor* conv_q, kda_tensor* conv_k,
                                 kda_tensor* conv_v, const kda_tensor* q, const kda_tensor* k,
                                 const kda_tensor* v, const kda_tensor* w_q, const kda_tensor* w_k,
                                 const kda_tensor* w_v, const kda_tensor* g, const kda_tensor* beta,
                                 const kda_tensor* out_gate, const kda_tensor* norm_weight, float scale,
                                 float eps, kda_tensor* out, void* stream);

/*
 * kda_recurrent_multi_step - n decode tokens per request in one call, with the
 * state read once and written back once (multi-token and speculative decoding).
 *
 * For every request and head it runs the recurrence above over tokens
 * 0 .. n-1 in order ("Kimi K3 核心算子拆解" (devpress.csdn.net) §2.3 for the
 * single step).  "Kimi K3 技术报告解读" (marsggbo.github.io) §9, on
 * speculative decoding with KDA, keeps only the draft tokens' inputs and
 * rebuilds the accepted tokens' state on chip by replaying them, verification
 * and write-back in one kernel; this call is that kernel: pass the previous
 * step's accepted tokens followed by the new drafts, with num_accepted = the
 * number of replayed tokens.  Token j's output uses the
 * state after tokens 0 .. j.  The state written back is the state after the
 * first num_accepted[request] tokens: a draft that was verified with outputs
 * (num_accepted = 0, nothing written) is committed by a second call without
 * outputs that replays the accepted tokens.
 *
 *   state        [N, H, d_k, d_v] f32, inner [d_k, d_v] contiguous; in/out
 *   q            [N, n, H, d_k] bf16 or f32, or NULL together with out
 *   k            [N, n, H, d_k]  same dtype as q
 *   v            [N, n, H, d_v]  same dtype as q
 *   g            [N, n, H, d_k]  f32, per-token log-decay
 *   beta         [N, n, H]       f32
 *   scale        finite float multiplying the read-out
 *   num_accepted [N] int32 on the device, or NULL (= n for every request);
 *                values are clamped to [0, n]; 0 leaves the state untouched
 *   out          [N, n, H, d_v]  k's dtype, or NULL (no outputs: only the
 *                accepted tokens are processed)
 *   stream       cudaStream_t as void*
 *
 * Errors as for kda_recurrent_step; q and out must both be given or both be
 * NULL.  n = 0 is a no-op.  The kernel takes the tokens four at a time (the
 * single step unrolled over each block of four, one pass over the state to
 * read and one to write per block, a block also ending where the accepted
 * tokens end), so the results equal n calls of kda_recurrent_step up to fp32
 * rounding.  n is meant to be small (draft lengths of a few tokens); any n
 * works.
 */
kda_status kda_recurrent_multi_step(kda_tensor* state, const kda_tensor* q, const kda_tensor* k,
                                    const kda_tensor* v, const kda_tensor* g, const kda_tensor* beta,
                                    float scale, const kda_tensor* num_accepted, kda_tensor* out,
                                    void* stream);

/*
 * kda_get_device_error - synchronises `stream`, then returns and clears the
 * current device's error word: KDA_OK, KDA_ERR_TIMEOUT (a bounded wait gave up;
 * reported first when several bits are set), KDA_ERR_DEVICE (bad cu_seqlens) or
 * KDA_ERR_DOMAIN (KDA_VALIDATE); KDA_ERR_CUDA if the synchronisation itself
 * failed.  The message of a non-OK result is available from
 * kda_last_error_message().
 */
kda_status kda_get_device_error(void* stream);

/* Static, human-readable name of a status code.  Never NULL. */
const char* kda_status_string(kda_status status);

/* Message of the last failed call on this host thread ("" if none).  Valid
 * until the next call into the library from this thread. */
const char* kda_last_error_message(void);

/*
 * Launch accounting, a measurement aid with no counterpart on the pages.
 *
 * kda_set_launch_events arms the calling host thread's next compute call
 * (kda_chunk_fwd, kda_chunk_fwd_noalloc, kda_fused_recurrent_fwd or
 * kda_recurrent_step), and that call only.  It records events[0] on its stream
 * just before its first kernel and events[i] just after its i-th kernel, as far
 * as `count` reaches.  The elapsed time between consecutive events is then the
 * device time of one kernel.
 *   events  array of `count` cudaEvent_t handles (as void*), created by the
 *           caller on the device of the call's stream; owned by the caller and
 *           needed only until the armed call returns.  NULL (with count 0)
 *           disarms.
 * Returns KDA_ERR_INVALID_ARG when count < 0, or events is NULL while
 * count > 0.  An event the runtime cannot record makes the armed call return
 * KDA_ERR_CUDA; the kernels it had enqueued by then stay enqueued.
 */
kda_status kda_set_launch_events(void* const* events, int count);

/* Number of kernels the calling thread's last compute call enqueued (0 when it
 * returned before launching any). */
int kda_last_launch_count(void);

/*
 * kda_test_stall_next_prefill - a testing hook with no counterpart on the pages:
 * it exercises the timeout path of the device-side waits without faulting or
 * hanging the GPU.  With on != 0 the calling host thread's next prefill call
 * (any kda_chunk_fwd* entry point; consumed by that call whatever it does) runs
 * its chunked serial kernel with the chunk-record copies suppressed and every
 * bounded wait cut to about 0.1 ms: the waits give up, the kernel stops issuing
 * work, drains what it issued, frees its tensor memory and returns, and
 * kda_get_device_error then reports KDA_ERR_TIMEOUT.  That call's outputs are
 * unspecified; later calls are unaffected.  on == 0 disarms.  Always KDA_OK.
 */
kda_status kda_test_stall_next_prefill(int on);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
