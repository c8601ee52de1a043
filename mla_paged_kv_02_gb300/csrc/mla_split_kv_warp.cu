// mla_split_kv_warp.cu -- first, plain split-KV attention kernel: one warp per
// (request, query row, split), streaming the request's pages straight from
// global memory with an online softmax.  Simple and obviously correct; the
// tensor-core kernel replaces it on the hot path.
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {

namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ float load_kv(const DecodeParams& p, int64_t idx, float kscale) {
  if (p.kv_fp8) {
    __nv_fp8_e4m3 v;
    v.__x = reinterpret_cast<const uint8_t*>(p.kv)[idx];
    return float(v) * kscale;
  }
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.kv)[idx]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
    split_kv_warp_kernel(const DecodeParams p) {
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int r = blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5);
  const int b = blockIdx.z;
  if (r >= p.rows) return;
  const int i = r / p.num_heads;  // query index; the head is r % num_heads
  const int64_t grow = (int64_t)b * p.rows + r;  // flat (b,i,h) row
  const int L = p.seq_lens[b];
  const float kscale = (p.kv_fp8 && p.kv_scale) ? *p.kv_scale : 1.0f;

  bool bad = !seq_len_ok(p, L);
  if (bad && lane == 0 && split == 0 && r == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, -1, L);

  float q[18];
  const __nv_bfloat16* qn = p.q_nope + grow * p.q_nope_stride;
  const __nv_bfloat16* qp = p.q_pe + grow * p.q_pe_stride;
#pragma unroll
  for (int k = 0; k < 16; ++k) q[k] = __bfloat162float(qn[lane + 32 * k]);
#pragma unroll
  for (int k = 0; k < 2; ++k) q[16 + k] = __bfloat162float(qp[lane + 32 * k]);

  float o[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) o[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float sc = p.softmax_scale * kscale;

  const int V = L - p.q_len + 1 + i;
  const int lo = split * p.chunk_tokens;
  const int hi = min(lo + p.chunk_tokens, V);
  if (!bad) {
    for (int t = lo; t < hi; ++t) {
      const int page = p.block_table[(int64_t)b * p.bt_stride + t / kPage];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, t / kPage, page);
        bad = true;
        break;
      }
      const int64_t base = ((int64_t)page * kPage + (t % kPage)) * kRow;
      float x[18];
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = load_kv(p, base + lane + 32 * k, 1.0f);
#pragma unroll
      for (int k = 0; k < 2; ++k) x[16 + k] = load_kv(p, base + kKvLora + lane + 32 * k, 1.0f);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 18; ++k) acc = fmaf(q[k], x[k], acc);
      const float s = warp_sum(acc) * sc;
      const float m_new = fmaxf(m, s);
      const float c = __expf(m - m_new);
      const float pt = __expf(s - m_new);
      l = l * c + pt;
#pragma unroll
      for (int k = 0; k < 16; ++k) o[k] = fmaf(o[k], c, pt * x[k] * kscale);
      m = m_new;
    }
  }

  float lse_v;
  if (bad) {
    lse_v = NAN;
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = NAN;
  } else if (hi <= lo) {
    lse_v = -INFINITY;  // empty split: weighs zero in the combine
  } else {
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] *= inv;
    lse_v = m + logf(l);
  }

  if (p.splits == 1) {
#pragma unroll
    for (int k = 0; k < 16; ++k) store_out(p, grow, lane + 32 * k, o[k]);
    if (p.lse && lane == 0) p.lse[grow] = lse_v;
  } else {
    float* dst = p.partials + (grow * p.splits + split) * kPartRow;
#pragma unroll
    for (int k = 0; k < 16; ++k) dst[lane + 32 * k] = o[k];
    if (lane == 0) dst[kKvLora] = lse_v;
  }
}

}  // namespace

cudaError_t launch_split_kv(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.splits, (p.rows + kWarpsPerCta - 1) / kWarpsPerCta, p.batch);
  split_kv_warp_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
