// mla_combine.cu -- LSE-weighted merge of split-KV partials.
//
// The partial layout [rows, splits, kv_lora_rank + 1] (512 normalised outputs,
// then the split's LSE) is the attn_logits layout of the Triton MLA split-KV
// path (vLLM PR #46819 summary, key code excerpt).  For each row:
//   M   = max_s lse_s
//   lse = M + ln sum_s exp(lse_s - M)
//   out = sum_s exp(lse_s - lse) * o_s
// Empty splits carry lse_s = -inf and weigh zero; their outputs are not read
// (the split kernel writes only the LSE of a split past a request's end).  A
// row whose first LSE is +inf belongs to a request with a single split, whose
// output the split kernel already wrote.  (A row whose splits are all
// empty, which only a sequence shard can have, gets out = 0 and lse = -inf).
// The same merge joins the partials of sequence shards gathered from several
// ranks, read with their own row and split strides.  One warp per row; each lane
// owns 16 of the 512 output columns, so every load of a split's 2 KB is a fully
// coalesced 128-byte transaction per lane group.  HBM-bound.
#include "common.cuh"

namespace mla {

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const DecodeParams p) {
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= (int64_t)p.batch * p.rows) return;
  const float* part = p.partials + row * p.part_row_stride;
  // +inf in the first partial's LSE: the request had a single split and the
  // split kernel wrote this row's out/lse itself.
  if (__ldcg(part + kKvLora) == INFINITY) return;
  merge_row(p, row, part, p.part_split_stride, p.splits, (p.out_fp8 && p.out_scale) ? *p.out_scale : 1.f);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.batch * p.rows;
  const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
  combine_kernel<<<blocks, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
