// mla_api.cu -- host side of the C ABI: split planner, argument validation,
// launches, and the sticky device error word.  Allocates nothing.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <numeric>
#include <queue>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#ifdef MLA_DEBUG
#include "mla_decode_debug.h"
#endif

using namespace mla;

namespace {

// Planner constants.  A 2-CTA cluster holds kRowsPerCta query rows (each CTA
// half of the 576 columns).  kSetupPages is the fixed cost of one cluster (Q
// staging, TMEM allocation, pipeline fill and epilogue) expressed in page-times.
constexpr int kRowsPerCta = 128;
constexpr int kCtasPerGroup = 2;
constexpr int kMaxSplits = 256;
constexpr double kSetupPages = 2.0;
// Fixed cost of the combine kernel (launch, and the dependent loads of a row's
// split LSEs), in page-times: about 10 us measured even for a tiny batch.
constexpr double kCombinePages = 8.0;
// The split kernel's grid is (2 * row_groups, splits, batch): the splits and
// the batch sit on gridDim.y and gridDim.z, whose hardware limit is 65535.
constexpr int kMaxGridYZ = 65535;
constexpr int kMaxRows = 4096;  // num_heads * q_len per request
// Token positions stay far from int32 overflow in split * chunk_tokens + chunk_tokens.
constexpr int kMaxSeqLen = 1 << 30;

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Length-aware planning (mla_decode_plan_lengths): costs in page-times of one
// cluster, measured on the split kernel.  A cluster's fixed cost (set-up, the
// drain after its last load, the epilogue) is about 14 us against about 1.1 us
// per page; a cluster whose split lies past its request's end exits at once.
constexpr double kClusterPages = 13.0;
constexpr double kEmptyClusterPages = 1.0;

// Bytes of fp32 split partials [batch, q_len, H, splits, 513]; none with one split.
size_t partial_bytes_for(int64_t batch, int64_t rows, int64_t splits) {
  return splits > 1 ? (size_t)(batch * rows * splits * (MLA_KV_LORA_RANK + 1)) * sizeof(float) : 0;
}

// A plan is usable only if every field is the planner's own arithmetic: the
// kernels size their writes from num_kv_splits, so a plan whose byte counts do
// not follow from its shape (edited after mla_decode_plan, or never planned)
// would let the split kernel write past the caller's workspace.
bool plan_ok(const mla_decode_plan_t* pl) {
  if (!(pl && pl->batch >= 1 && pl->batch <= kMaxGridYZ && pl->num_heads >= 1 && pl->q_len >= 1 &&
        pl->q_len <= MLA_MAX_Q_LEN && (int64_t)pl->num_heads * pl->q_len <= kMaxRows &&
        pl->page_size == MLA_PAGE_SIZE && pl->max_seq_len >= pl->q_len && pl->num_kv_splits >= 1 &&
        pl->num_kv_splits <= kMaxGridYZ && pl->chunk_tokens >= MLA_PAGE_SIZE &&
        pl->chunk_tokens % MLA_PAGE_SIZE == 0 && pl->rows_per_cta == kRowsPerCta &&
        pl->row_groups == ceil_div((int64_t)pl->num_heads * pl->q_len, kRowsPerCta) &&
        (pl->kv_dtype == MLA_KV_BF16 || pl->kv_dtype == MLA_KV_FP8_E4M3) &&
        pl->max_seq_len <= kMaxSeqLen && pl->chunk_tokens <= pl->max_seq_len + MLA_PAGE_SIZE - 1 &&
        (int64_t)pl->num_kv_splits * pl->chunk_tokens >= pl->max_seq_len &&
        (int64_t)(pl->num_kv_splits - 1) * pl->chunk_tokens < pl->max_seq_len))
    return false;
  const size_t part = partial_bytes_for(pl->batch, (int64_t)pl->num_heads * pl->q_len, pl->num_kv_splits);
  return pl->partial_bytes == part && pl->workspace_bytes == MLA_WORKSPACE_HEADER_BYTES + part;
}

#ifdef MLA_DEBUG
uint64_t g_debug_wait_limit_ns = 0;  // 0: the kernels' built-in limit
#endif

}  // namespace

bool mla::plan_valid(const mla_decode_plan_t* pl) { return plan_ok(pl); }

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// q_fp8: the query is e4m3 codes (1 byte each), which also admits an FP8
// output; otherwise it is bf16 and the output bf16 or fp32.
mla_status_t fill_params(const mla_decode_plan_t* pl, const void* q_nope, int64_t q_nope_row_stride,
                         const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
                         int num_pages, const int32_t* block_table, int block_table_stride,
                         const int32_t* seq_lens, float softmax_scale, const float* kv_scale,
                         void* out, mla_out_dtype_t out_dtype, float* lse, void* workspace,
                         size_t workspace_bytes, DecodeParams* p, bool q_fp8 = false) {
  if (!plan_ok(pl)) return MLA_ERR_INVALID_ARG;
  if (!q_nope || !q_pe || !kv_cache || !block_table || !seq_lens || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  // Row strides: whole rows, and 16-byte multiples (the TMA stride rule).
  const int64_t stride_mult = q_fp8 ? 16 : 8;
  if (q_nope_row_stride < MLA_KV_LORA_RANK || q_pe_row_stride < MLA_QK_ROPE_DIM ||
      q_nope_row_stride % stride_mult || q_pe_row_stride % stride_mult)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 16) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || (int64_t)num_pages * MLA_PAGE_SIZE > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (block_table_stride < ceil_div(pl->max_seq_len, MLA_PAGE_SIZE)) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_OUT_BF16 && out_dtype != MLA_OUT_FP32 && !(q_fp8 && out_dtype == MLA_OUT_FP8_E4M3))
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < pl->workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;

  memset(p, 0, sizeof *p);
  p->q_fp8 = q_fp8;
  p->out_fp8 = out_dtype == MLA_OUT_FP8_E4M3;
  p->q_nope = q_nope;
  p->q_nope_stride = q_nope_row_stride;
  p->q_pe = q_pe;
  p->q_pe_stride = q_pe_row_stride;
  p->kv = kv_cache;
  p->num_pages = num_pages;
  p->kv_fp8 = pl->kv_dtype == MLA_KV_FP8_E4M3;
  p->block_table = block_table;
  p->bt_stride = block_table_stride;
  p->seq_lens = seq_lens;
  p->softmax_scale = softmax_scale;
  p->kv_scale = kv_scale;
  p->out = out;
  p->out_fp32 = out_dtype == MLA_OUT_FP32;
  p->out_stride = MLA_KV_LORA_RANK;
  p->lse = lse;
  p->lse_stride = 1;
  p->err = static_cast<int32_t*>(workspace);
  p->partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + MLA_WORKSPACE_HEADER_BYTES);
  p->batch = pl->batch;
  p->num_heads = pl->num_heads;
  p->q_len = pl->q_len;
  p->rows = pl->num_heads * pl->q_len;
  p->max_seq_len = pl->max_seq_len;
  p->splits = pl->num_kv_splits;
  p->chunk_tokens = pl->chunk_tokens;
  p->rows_per_cta = pl->rows_per_cta;
  p->row_groups = pl->row_groups;
  // Longest requests first, when more clusters than the GPU holds at once wait
  // to start (with a single wave the order does not matter).
  const int64_t clusters = (int64_t)pl->batch * pl->row_groups * pl->num_kv_splits;
  p->order_by_length = pl->batch <= kMaxOrderedBatch && clusters > pl->num_sms / 2;
#ifdef MLA_DEBUG
  p->wait_limit_ns = g_debug_wait_limit_ns;
#endif
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_plan(int batch, int num_heads, int q_len, int max_seq_len, int page_size,
                             mla_kv_dtype_t kv_dtype, int num_sms, int force_splits,
                             mla_decode_plan_t* plan) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  memset(plan, 0, sizeof *plan);
  if (batch < 1 || num_heads < 1 || q_len < 1 || max_seq_len < 1 || force_splits < 0)
    return MLA_ERR_INVALID_ARG;
  if (page_size != MLA_PAGE_SIZE || q_len > MLA_MAX_Q_LEN) return MLA_ERR_UNSUPPORTED;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  if (max_seq_len < q_len) return MLA_ERR_INVALID_ARG;
  if ((int64_t)num_heads * q_len > kMaxRows || batch > kMaxGridYZ || max_seq_len > kMaxSeqLen)
    return MLA_ERR_UNSUPPORTED;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
  }
  const int rows = num_heads * q_len;
  const int row_groups = ceil_div(rows, kRowsPerCta);
  const int pages = ceil_div(max_seq_len, MLA_PAGE_SIZE);
  const double page_bytes = (kv_dtype == MLA_KV_FP8_E4M3 ? 1.0 : 2.0) * MLA_KV_ROW * MLA_PAGE_SIZE;

  int splits = 1;
  if (force_splits > 0) {
    splits = force_splits < pages ? force_splits : pages;
    if (splits > kMaxGridYZ) splits = kMaxGridYZ;
  } else {
    // Smallest modelled time: whole waves of one-CTA-per-SM work, each CTA paying
    // its pages plus a fixed set-up, plus the partial write+read and the combine
    // kernel's fixed cost when there is more than one split, all in per-SM
    // page-times.
    double best = 1e300;
    const int smax = pages < kMaxSplits ? pages : kMaxSplits;
    for (int s = 1; s <= smax; ++s) {
      const int64_t ctas = (int64_t)batch * row_groups * kCtasPerGroup * s;
      const int64_t waves = (ctas + num_sms - 1) / num_sms;
      const int ppc = ceil_div(pages, s);
      double cost = (double)waves * (ppc + kSetupPages);
      if (s > 1) {
        const double pbytes = 2.0 * batch * rows * (double)s * (MLA_KV_LORA_RANK + 1) * 4.0;
        cost += pbytes / (num_sms * page_bytes) + kCombinePages;
      }
      if (cost < best * (1.0 - 1e-9)) {
        best = cost;
        splits = s;
      }
    }
  }
  const int chunk_pages = ceil_div(pages, splits);
  splits = ceil_div(pages, chunk_pages);  // no split lies wholly past max_seq_len

  plan->batch = batch;
  plan->num_heads = num_heads;
  plan->q_len = q_len;
  plan->max_seq_len = max_seq_len;
  plan->page_size = page_size;
  plan->kv_dtype = kv_dtype;
  plan->num_sms = num_sms;
  plan->num_kv_splits = splits;
  plan->chunk_tokens = chunk_pages * MLA_PAGE_SIZE;
  plan->rows_per_cta = kRowsPerCta;
  plan->row_groups = row_groups;
  plan->partial_bytes = partial_bytes_for(batch, rows, splits);
  plan->workspace_bytes = MLA_WORKSPACE_HEADER_BYTES + plan->partial_bytes;
  return MLA_OK;
}

mla_status_t mla_workspace_init(void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!workspace || workspace_bytes < MLA_WORKSPACE_HEADER_BYTES) return MLA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, MLA_WORKSPACE_HEADER_BYTES, (cudaStream_t)cuda_stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_split_kv(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                          const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
                          int num_pages, const int32_t* block_table, int block_table_stride,
                          const int32_t* seq_lens, float softmax_scale, const float* kv_scale,
                          void* out, mla_out_dtype_t out_dtype, float* lse, void* workspace,
                          size_t workspace_bytes, void* cuda_stream) {
  DecodeParams p;
  mla_status_t st = fill_params(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache,
                                num_pages, block_table, block_table_stride, seq_lens, softmax_scale,
                                kv_scale, out, out_dtype, lse, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  if (launch_split_kv(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_decode_plan_lengths(int batch, int num_heads, int q_len, const int32_t* seq_lens,
                                     int page_size, mla_kv_dtype_t kv_dtype, int num_sms,
                                     mla_decode_plan_t* plan) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  memset(plan, 0, sizeof *plan);
  if (!seq_lens || batch < 1) return MLA_ERR_INVALID_ARG;
  int max_len = q_len;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < q_len) return MLA_ERR_INVALID_ARG;
    max_len = std::max(max_len, (int)seq_lens[b]);
  }
  // The length-blind plan for the longest request: its split count bounds the
  // candidates (uneven lengths only ever want fewer splits) and its checks
  // apply unchanged.
  mla_decode_plan_t uni;
  mla_status_t st = mla_decode_plan(batch, num_heads, q_len, max_len, page_size, kv_dtype, num_sms, 0, &uni);
  if (st != MLA_OK) return st;
  const int64_t rows = (int64_t)num_heads * q_len;
  const int rg = uni.row_groups;
  const int slots = std::max(1, uni.num_sms / kCtasPerGroup);
  const int pages = ceil_div(max_len, MLA_PAGE_SIZE);
  const double page_bytes = (kv_dtype == MLA_KV_FP8_E4M3 ? 1.0 : 2.0) * MLA_KV_ROW * MLA_PAGE_SIZE;
  std::vector<int> req_pages(batch), order(batch);
  for (int b = 0; b < batch; ++b) req_pages[b] = ceil_div(seq_lens[b], MLA_PAGE_SIZE);
  std::iota(order.begin(), order.end(), 0);
  std::vector<int> by_len = order;  // the kernel's longest-first order (ties by index)
  std::stable_sort(by_len.begin(), by_len.end(), [&](int a, int c) { return seq_lens[a] > seq_lens[c]; });

  // Each candidate split count: the clusters in the order the hardware starts
  // them (grid order, requests longest first when the kernel ranks them), each
  // taken by the cluster slot that frees first; plus the combine's partial
  // traffic and fixed cost when any request has more than one split.
  int best_s = uni.num_kv_splits;
  double best = 1e300;
  for (int s = 1; s <= uni.num_kv_splits; ++s) {
    const int chunk = ceil_div(pages, s);
    if (ceil_div(pages, chunk) != s) continue;  // not a distinct plan
    const bool lpt = batch <= kMaxOrderedBatch && (int64_t)batch * rg * s > slots;
    const std::vector<int>& seq = lpt ? by_len : order;
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < slots; ++i) free_at.push(0.0);
    double part_bytes = 0.0;
    for (int b : seq) {
      const int sb = std::max(1, std::min(s, ceil_div(req_pages[b], chunk)));
      if (sb > 1) part_bytes += 2.0 * rows * sb * (MLA_KV_LORA_RANK + 1) * 4.0;
      for (int k = 0; k < s; ++k) {
        const double cost = k < sb ? kClusterPages + std::min(chunk, req_pages[b] - k * chunk) : kEmptyClusterPages;
        for (int r = 0; r < rg; ++r) {
          const double t = free_at.top();
          free_at.pop();
          free_at.push(t + cost);
        }
      }
    }
    double makespan = 0.0;
    while (!free_at.empty()) {
      makespan = std::max(makespan, free_at.top());
      free_at.pop();
    }
    if (part_bytes > 0) makespan += part_bytes / (uni.num_sms * page_bytes) + kCombinePages;
    if (makespan < best * (1.0 - 1e-9)) {
      best = makespan;
      best_s = s;
    }
  }
  return mla_decode_plan(batch, num_heads, q_len, max_len, page_size, kv_dtype, uni.num_sms, best_s, plan);
}

}  // extern "C"

namespace {

// The combine of the workspace partials into out (row stride out_stride) and
// lse (stride lse_stride).
mla_status_t combine_workspace(const mla_decode_plan_t* plan, void* out, mla_out_dtype_t out_dtype,
                               int64_t out_stride, float* lse, int64_t lse_stride, const void* workspace,
                               size_t workspace_bytes, void* cuda_stream, const float* out_scale = nullptr) {
  if (!plan_ok(plan) || !out || !workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_OUT_BF16 && out_dtype != MLA_OUT_FP32 &&
      !(out_dtype == MLA_OUT_FP8_E4M3 && out_stride == MLA_KV_LORA_RANK))
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (plan->num_kv_splits == 1) return MLA_OK;
  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.out = out;
  p.out_fp32 = out_dtype == MLA_OUT_FP32;
  p.out_fp8 = out_dtype == MLA_OUT_FP8_E4M3;
  p.out_scale = out_scale;
  p.out_stride = out_stride;
  p.lse = lse;
  p.lse_stride = lse_stride;
  p.partials = reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(workspace)) +
                                        MLA_WORKSPACE_HEADER_BYTES);
  p.batch = plan->batch;
  p.num_heads = plan->num_heads;
  p.q_len = plan->q_len;
  p.rows = plan->num_heads * plan->q_len;
  p.splits = plan->num_kv_splits;
  p.part_row_stride = (int64_t)p.splits * kPartRow;
  p.part_split_stride = kPartRow;
  if (launch_combine(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_combine(const mla_decode_plan_t* plan, void* out, mla_out_dtype_t out_dtype,
                         float* lse, const void* workspace, size_t workspace_bytes,
                         void* cuda_stream) {
  return combine_workspace(plan, out, out_dtype, MLA_KV_LORA_RANK, lse, 1, workspace, workspace_bytes,
                           cuda_stream);
}

mla_status_t mla_decode_shard(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                              const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache, int num_pages,
                              const int32_t* block_table, int block_table_stride, const int32_t* shard_lens,
                              const int32_t* shard_start, const int32_t* seq_lens, float softmax_scale,
                              const float* kv_scale, float* shard_partial, void* workspace,
                              size_t workspace_bytes, void* cuda_stream) {
  if (!shard_lens || !shard_start || !seq_lens || !shard_partial || !aligned(shard_partial, 4))
    return MLA_ERR_INVALID_ARG;
  DecodeParams p;
  mla_status_t st = fill_params(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_pages,
                                block_table, block_table_stride, shard_lens, softmax_scale, kv_scale,
                                shard_partial, MLA_OUT_FP32, shard_partial + MLA_KV_LORA_RANK, workspace,
                                workspace_bytes, &p);
  if (st != MLA_OK) return st;
  // One 513-wide fp32 row per query row: the 512 outputs, then the LSE.
  p.out_stride = kPartRow;
  p.lse_stride = kPartRow;
  p.kv_start = shard_start;
  p.total_lens = seq_lens;
  if (launch_split_kv(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return combine_workspace(plan, shard_partial, MLA_OUT_FP32, kPartRow, shard_partial + MLA_KV_LORA_RANK,
                           kPartRow, workspace, workspace_bytes, cuda_stream);
}

mla_status_t mla_decode_fp8(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                            const void* q_pe, int64_t q_pe_row_stride, const float* q_scale, const void* kv_cache,
                            int num_pages, const int32_t* block_table, int block_table_stride,
                            const int32_t* seq_lens, float softmax_scale, const float* kv_scale, void* out,
                            mla_out_dtype_t out_dtype, const float* out_scale, float* lse, void* workspace,
                            size_t workspace_bytes, void* cuda_stream) {
  if (plan && plan->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  DecodeParams p;
  mla_status_t st = fill_params(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_pages,
                                block_table, block_table_stride, seq_lens, softmax_scale, kv_scale, out, out_dtype,
                                lse, workspace, workspace_bytes, &p, /*q_fp8=*/true);
  if (st != MLA_OK) return st;
  p.q_scale = q_scale;
  p.out_scale = out_scale;
  if (launch_split_kv(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return combine_workspace(plan, out, out_dtype, MLA_KV_LORA_RANK, lse, 1, workspace, workspace_bytes, cuda_stream,
                           out_scale);
}

mla_status_t mla_combine_shards(int64_t rows, int num_shards, const float* shard_partials, void* out,
                                mla_out_dtype_t out_dtype, float* lse, void* cuda_stream) {
  if (rows < 1 || rows > INT32_MAX || num_shards < 1 || !shard_partials || !out) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_OUT_BF16 && out_dtype != MLA_OUT_FP32) return MLA_ERR_INVALID_ARG;
  if (!aligned(shard_partials, 4) || !aligned(out, 4)) return MLA_ERR_INVALID_ARG;
  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.out = out;
  p.out_fp32 = out_dtype == MLA_OUT_FP32;
  p.out_stride = MLA_KV_LORA_RANK;
  p.lse = lse;
  p.lse_stride = 1;
  p.partials = const_cast<float*>(shard_partials);
  p.batch = 1;
  p.rows = (int)rows;
  p.splits = num_shards;
  p.part_row_stride = kPartRow;
  p.part_split_stride = rows * kPartRow;
  if (launch_combine(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_decode(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                        const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
                        int num_pages, const int32_t* block_table, int block_table_stride,
                        const int32_t* seq_lens, float softmax_scale, const float* kv_scale,
                        void* out, mla_out_dtype_t out_dtype, float* lse, void* workspace,
                        size_t workspace_bytes, void* cuda_stream) {
  mla_status_t st = mla_split_kv(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache,
                                 num_pages, block_table, block_table_stride, seq_lens,
                                 softmax_scale, kv_scale, out, out_dtype, lse, workspace,
                                 workspace_bytes, cuda_stream);
  if (st != MLA_OK) return st;
  return mla_combine(plan, out, out_dtype, lse, workspace, workspace_bytes, cuda_stream);
}

mla_status_t mla_decode_varlen(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                               const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
                               int num_pages, const int32_t* block_table, int block_table_stride,
                               const int32_t* seq_lens, const int32_t* q_lens, float softmax_scale,
                               const float* kv_scale, void* out, mla_out_dtype_t out_dtype, float* lse,
                               void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!q_lens) return MLA_ERR_INVALID_ARG;
  DecodeParams p;
  mla_status_t st = fill_params(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache,
                                num_pages, block_table, block_table_stride, seq_lens, softmax_scale,
                                kv_scale, out, out_dtype, lse, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  p.q_lens = q_lens;
  if (launch_split_kv(p, (cudaStream_t)cuda_stream) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_combine(plan, out, out_dtype, lse, workspace, workspace_bytes, cuda_stream);
}

mla_status_t mla_decode_check_error(void* workspace, void* cuda_stream, int32_t info[4]) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  int32_t h[4] = {0, 0, 0, 0};
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyAsync(h, workspace, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (info) memcpy(info, h, sizeof h);
  if (h[kHdrCode] != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof h, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    return h[kHdrCode] == MLA_ERR_TIMEOUT ? MLA_ERR_TIMEOUT : MLA_ERR_DEVICE_INPUT;
  }
  return MLA_OK;
}

#ifdef MLA_DEBUG
mla_status_t mla_debug_set_wait_limit_ns(uint64_t ns) {
  g_debug_wait_limit_ns = ns;
  return MLA_OK;
}
#endif

const char* mla_status_string(mla_status_t status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_INPUT: return "MLA_ERR_DEVICE_INPUT";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
  }
  return "MLA_ERR_UNKNOWN";
}

}  // extern "C"
