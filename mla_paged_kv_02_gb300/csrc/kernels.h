// kernels.h -- launchers the C-ABI layer calls (one translation unit each) and
// the plan check the entry points share.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// Split-KV attention stage (paged gather, QK^T, masked online softmax, PV,
// split epilogue): writes out/lse directly for one split, partials otherwise.
cudaError_t launch_split_kv(const DecodeParams& p, cudaStream_t stream);

// LSE-weighted combine of the split partials into out/lse.
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);

// True when every field of the plan follows from its shape by the planner's own
// arithmetic (host only, touches no GPU).
bool plan_valid(const mla_decode_plan_t* pl);

}  // namespace mla
