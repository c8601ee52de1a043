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

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// kGathered: shard partials [splits, rows, 513] read with the strides in p;
// otherwise the workspace layout [rows, splits, 513] with constant strides.
template <bool kGathered>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const DecodeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= (int64_t)p.batch * p.rows) return;
  const float* part = p.partials + row * (kGathered ? p.part_row_stride : (int64_t)p.splits * kPartRow);
  const int64_t sstride = kGathered ? p.part_split_stride : kPartRow;
  const float osc = (p.out_fp8 && p.out_scale) ? *p.out_scale : 1.f;

  if (p.splits <= 32) {
    // Lane s holds split s's LSE and, once the total is known, its weight.
    // The outputs of four splits are loaded at a time (64 loads per lane in
    // flight, the weights by shuffle), so a row costs one dependent round trip
    // per four splits instead of two per split.
    const float lv = lane < p.splits ? part[(int64_t)lane * sstride + kKvLora] : -INFINITY;
    // +inf in the first partial's LSE: the request had a single split and the
    // split kernel wrote this row's out/lse itself.
    if (__shfl_sync(0xffffffffu, lv, 0) == INFINITY) return;
    const bool nan_seen = __any_sync(0xffffffffu, lv != lv);
    const float M = warp_max(lv);
    const float acc = warp_sum(lv == -INFINITY ? 0.f : __expf(lv - M));
    const float lse = (M == -INFINITY || nan_seen) ? (nan_seen ? NAN : -INFINITY) : M + logf(acc);
    const float wl = (lv == -INFINITY || nan_seen || M == -INFINITY) ? 0.f : __expf(lv - lse);
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = nan_seen ? NAN : 0.f;
    if (!nan_seen) {
      for (int s0 = 0; s0 < p.splits; s0 += 4) {
        float w[4], v[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = __shfl_sync(0xffffffffu, wl, (s0 + j) & 31);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // Splits past the last, and empty ones (weight 0, outputs not read).
          const bool use = s0 + j < p.splits && w[j] != 0.f;
          const float* ps = part + (int64_t)(s0 + j) * sstride + lane;
#pragma unroll
          for (int k = 0; k < 16; ++k) v[j][k] = use ? ps[32 * k] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float wj = s0 + j < p.splits ? w[j] : 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) o[k] = fmaf(wj, v[j][k], o[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) store_out(p, row, lane + 32 * k, o[k], osc);
    if (p.lse && lane == 0) p.lse[row * p.lse_stride] = lse;
    return;
  }

  // More than 32 splits.  Pass 1: the largest split LSE (NaN marks a request
  // the split kernel rejected).
  float M = -INFINITY;
  bool nan_seen = false;
  bool single = false;
  for (int s = lane; s < p.splits; s += 32) {
    const float v = part[(int64_t)s * sstride + kKvLora];
    // +inf in the first partial's LSE: the request had a single split and the
    // split kernel wrote this row's out/lse itself.
    single |= (s == 0) & (v == INFINITY);
    nan_seen |= (v != v);
    M = fmaxf(M, v);
  }
  if (__any_sync(0xffffffffu, single)) return;
  M = warp_max(M);
  nan_seen = __any_sync(0xffffffffu, nan_seen);

  float acc = 0.f;
  for (int s = lane; s < p.splits; s += 32) {
    const float v = part[(int64_t)s * sstride + kKvLora];
    acc += (v == -INFINITY) ? 0.f : __expf(v - M);
  }
  acc = warp_sum(acc);
  const float lse = (M == -INFINITY || nan_seen) ? (nan_seen ? NAN : -INFINITY) : M + logf(acc);

  float o[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) o[k] = 0.f;
  if (!nan_seen && M != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float* ps = part + (int64_t)s * sstride;
      const float v = ps[kKvLora];
      if (v == -INFINITY) continue;
      const float w = __expf(v - lse);
#pragma unroll
      for (int k = 0; k < 16; ++k) o[k] = fmaf(w, ps[lane + 32 * k], o[k]);
    }
  } else if (nan_seen) {
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = NAN;
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) store_out(p, row, lane + 32 * k, o[k], osc);
  if (p.lse && lane == 0) p.lse[row * p.lse_stride] = lse;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.batch * p.rows;
  const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
  if (p.part_split_stride == kPartRow && p.part_row_stride == (int64_t)p.splits * kPartRow)
    combine_kernel<false><<<blocks, kWarps * 32, 0, stream>>>(p);
  else
    combine_kernel<true><<<blocks, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
