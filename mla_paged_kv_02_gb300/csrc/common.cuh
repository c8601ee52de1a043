// common.cuh -- kernel parameter block and small device helpers shared by the
// split-KV attention kernel, the combine kernel and the host launcher.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_decode.h"

namespace mla {

constexpr int kKvLora = MLA_KV_LORA_RANK;  // 512: c_kv width, also the output width
constexpr int kRope = MLA_QK_ROPE_DIM;     // 64: k_pe / q_pe width
constexpr int kRow = MLA_KV_ROW;           // 576 entries per cached token
constexpr int kPage = MLA_PAGE_SIZE;       // 64 tokens per page
constexpr int kPartRow = kKvLora + 1;      // one split partial: 512 outputs + LSE

// Workspace header layout (int32 words).  The first word is the sticky error
// code (0 = none); the next three describe the first error seen.
constexpr int kHdrCode = 0, kHdrRequest = 1, kHdrIndex = 2, kHdrValue = 3;

struct DecodeParams {
  const void* q_nope;     // bf16, or e4m3 codes when q_fp8
  int64_t q_nope_stride;  // elements between consecutive (b,i,h) rows
  const void* q_pe;
  int64_t q_pe_stride;
  int q_fp8;              // the query is e4m3 codes times *q_scale (FP8 cache only)
  const float* q_scale;   // device scalar or nullptr (1)
  const void* kv;  // [num_pages, 64, 576] bf16 or e4m3 bytes
  int num_pages;
  int kv_fp8;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;  // [B] tokens of request b in this cache (a shard's own count under DCP)
  const int32_t* q_lens;  // [B] per-request number of query tokens (1..q_len), or nullptr: all q_len
  // Sequence shard (DCP): absolute position of this cache's first token of
  // request b, and the request's whole length (the causal mask is on absolute
  // positions).  nullptr: the cache holds the whole request from position 0.
  const int32_t* kv_start;
  const int32_t* total_lens;
  float softmax_scale;
  const float* kv_scale;  // device scalar or nullptr
  void* out;              // [B*R rows] of 512 bf16, fp32 or e4m3, out_stride elements apart
  int out_fp32;
  int out_fp8;            // e4m3 code of out / *out_scale (round to nearest even, saturating)
  const float* out_scale; // device scalar or nullptr (1)
  int64_t out_stride;     // 512, or 513 when out/lse are the two parts of a 513-wide partial row
  float* lse;       // [B*R] lse_stride apart, or nullptr
  int64_t lse_stride;
  float* partials;  // [B*R, splits, 513] fp32 (splits > 1)
  // Combine only: element distance between rows and between splits of the
  // partials it reads ([rows, splits, 513] in the workspace; [splits, rows, 513]
  // for gathered shard partials).
  int64_t part_row_stride, part_split_stride;
  int32_t* err;     // workspace header
  int batch, num_heads, q_len, rows;  // rows = num_heads * q_len per request
  int max_seq_len, splits, chunk_tokens, rows_per_cta, row_groups;
  int order_by_length;  // clusters take the requests longest first (see kMaxOrderedBatch)
  // Limit of every bounded device wait in ns (0: the built-in 1 s).  Only a
  // library built with MLA_DEBUG lets a caller set it (to test the timeout path).
  uint64_t wait_limit_ns;
};

// Batches up to this size are ranked by length inside the split kernel.
constexpr int kMaxOrderedBatch = 1024;

// Records the first device-side error of a call sequence (sticky until read).
__device__ __forceinline__ void report_error(int32_t* err, int code, int request, int index,
                                             int value) {
  if (atomicCAS(err + kHdrCode, 0, code) == 0) {
    err[kHdrRequest] = request;
    err[kHdrIndex] = index;
    err[kHdrValue] = value;
    __threadfence();
  }
}

// out / out_scale as an e4m3 code: round to nearest even, saturating to +-448;
// NaN stays NaN (0x7F / 0xFF).
__device__ __forceinline__ uint8_t to_e4m3(float v, float out_scale) {
  return (uint8_t)__nv_cvt_float_to_fp8(v / out_scale, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ void store_out(const DecodeParams& p, int64_t row, int d, float v, float out_scale) {
  if (p.out_fp32)
    reinterpret_cast<float*>(p.out)[row * p.out_stride + d] = v;
  else if (p.out_fp8)
    reinterpret_cast<uint8_t*>(p.out)[row * p.out_stride + d] = to_e4m3(v, out_scale);
  else
    reinterpret_cast<__nv_bfloat16*>(p.out)[row * p.out_stride + d] = __float2bfloat16_rn(v);
}

}  // namespace mla
