// Internal interface of the chunked backward (kda_backward_chunk.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "kda_internal.h"

namespace kda {

// Bytes of device scratch the chunked backward needs for these sizes (varlen when
// cu_seqlens is set); 0 when the chunk count does not fit an int (unsupported).
size_t chunk_backward_workspace_bytes(const PrefillArgs& a);

// Gradients as kda_backward computes them, by the chunked form: ws holds
// chunk_backward_workspace_bytes(ba.f) bytes of device memory used only by work
// enqueued on s.  ba.ck, ba.scr and ba.part are not used.
cudaError_t launch_chunk_backward(const BackwardArgs& ba, void* ws, cudaStream_t s);

}  // namespace kda
