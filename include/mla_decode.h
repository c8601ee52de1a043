/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA paged-KV decode library.
 *
 * Operation (multi-head latent attention decode in absorbed form, DeepSeek-R1
 * dims; the dims and uniform query length come from the vLLM PR #41778
 * "TOKENSPEED_MLA" summary, risks 4 and 6; the split partial layout of width
 * kv_lora_rank + 1 from the vLLM PR #46819 "Triton MLA attn logits
 * preallocation" summary, key code excerpt):
 *
 *   Each cached token is a 576-entry row x = c_kv (512) | k_pe (64), stored in
 *   pages of 64 tokens.  For request b with L = seq_lens[b] tokens (the q_len
 *   new tokens included), query index i in [0, q_len) and head h:
 *     visible V = L - q_len + 1 + i        (causal inside the q_len block)
 *     s_t   = softmax_scale * (q_nope . c_kv_t + q_pe . k_pe_t),   t < V
 *     out   = sum_t softmax(s)_t * c_kv_t    (512 entries)
 *     lse   = ln sum_t exp(s_t)
 *   With an FP8-E4M3 cache, x = e4m3 * kv_scale (one per-tensor scale).
 *
 * Row order everywhere: rows are (b, i, h) with flat index (b*q_len + i)*H + h.
 *
 * Ownership: the caller owns every buffer, including the workspace.  Every
 * entry point except mla_decode_noalloc allocates no device memory, keeps no
 * state between calls and caches no scale (a stale cached scale and a leaked
 * per-device workspace are the two risks the TokenSpeed MLA review flags).
 * mla_decode_noalloc is the one exception: it works in a fixed array that the
 * library's device image reserves on every GPU that loads it (see its block
 * below for the size and the sharing rules).  All device work is asynchronous
 * on the caller's stream; no entry point but mla_decode_check_error
 * synchronises.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,         /* a host-checkable argument is wrong            */
    MLA_ERR_UNSUPPORTED = 2,         /* dims/page size/q_len outside what is built    */
    MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < plan->workspace_bytes       */
    MLA_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed             */
    MLA_ERR_DEVICE_INPUT = 5,        /* device-side check: bad seq_len or page index  */
    MLA_ERR_TIMEOUT = 6              /* a bounded device wait gave up                 */
} mla_status_t;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype_t;
/* MLA_OUT_FP8_E4M3 (e4m3 codes of out / out_scale) only through mla_decode_fp8. */
typedef enum { MLA_OUT_BF16 = 0, MLA_OUT_FP32 = 1, MLA_OUT_FP8_E4M3 = 2 } mla_out_dtype_t;

/* Fixed geometry of the latent cache (DeepSeek-R1). */
#define MLA_KV_LORA_RANK 512
#define MLA_QK_ROPE_DIM 64
#define MLA_KV_ROW (MLA_KV_LORA_RANK + MLA_QK_ROPE_DIM)
#define MLA_PAGE_SIZE 64
#define MLA_MAX_Q_LEN 8
#define MLA_WORKSPACE_HEADER_BYTES 256

typedef struct {
    int batch, num_heads, q_len, max_seq_len, page_size, kv_dtype, num_sms;
    int num_kv_splits;   /* splits per request (>= 1)                                   */
    int chunk_tokens;    /* tokens per split, a multiple of page_size                   */
    int rows_per_cta;    /* query rows one CTA holds                                    */
    int row_groups;      /* ceil(num_heads * q_len / rows_per_cta)                      */
    int reserved[3];
    size_t partial_bytes;   /* fp32 split partials [B, q_len, H, splits, 513]; 0 if 1 split */
    size_t workspace_bytes; /* header + partials                                        */
} mla_decode_plan_t;

/*
 * mla_decode_plan -- host-only integer planning step (vLLM PR #46819 summary:
 * one split-count function shared by workspace reservation and the call, so
 * that a workspace reserved once at the worst case never has to grow).
 *
 *   batch, num_heads, q_len : problem shape; q_len in 1..8 (uniform per call)
 *   max_seq_len             : an upper bound on every seq_lens[b] of the calls
 *                             that will use this plan (>= q_len)
 *   page_size               : must be 64
 *   num_sms                 : SMs to plan for; 0 = query the current device
 *   force_splits            : 0 = choose; > 0 = use this many splits (clamped
 *                             so every split holds at least one page)
 *   plan                    : out
 *
 * Splits are chosen so that batch * row_groups * splits CTAs fill whole waves
 * of the SMs while each split keeps enough pages to amortise its set-up, and
 * the partial bytes stay small next to the KV bytes (the TokenSpeed summary,
 * implementation step 1, sizes its partials from the SM count for the same
 * reason).  Returns MLA_ERR_UNSUPPORTED for page_size != 64, q_len outside
 * 1..8, num_heads * q_len > 4096, batch > 65535 (the batch is a grid
 * dimension) or max_seq_len > 2^30, and MLA_ERR_INVALID_ARG for non-positive
 * sizes.  Touches no GPU when num_sms > 0.
 *
 * Every entry point that takes a plan re-derives its byte counts and split
 * geometry from its shape and returns MLA_ERR_INVALID_ARG, before any launch,
 * for a plan that was edited after mla_decode_plan filled it in.
 */
mla_status_t mla_decode_plan(int batch, int num_heads, int q_len, int max_seq_len, int page_size,
                             mla_kv_dtype_t kv_dtype, int num_sms, int force_splits,
                             mla_decode_plan_t* plan);

/*
 * mla_decode_plan_lengths -- the same plan, with the split count chosen from
 * the batch's own lengths rather than from an upper bound (a balanced split
 * scheduler for uneven lengths, the TokenSpeed MLA summary's scheduler item).
 * Host-only.
 *
 *   seq_lens : host int32 [batch], the lengths the call will see (q_len <= L_b)
 *   other arguments as mla_decode_plan (max_seq_len = the largest seq_lens[b])
 *
 * Every candidate split count up to the length-blind plan's for the longest
 * request is tried on a model of the split kernel: each (request, split, row
 * group) cluster costs a fixed 13 page-times plus its pages (1 for a split
 * past its request's end), clusters start in the kernel's order (requests
 * longest first when it ranks them) on the first cluster slot to free, and
 * partial traffic plus the combine's fixed cost are added when a request has
 * more than one split; the smallest modelled time wins (ties to fewer
 * splits).  With equal lengths this is the length-blind choice or one with
 * fewer waves; with uneven lengths the long requests dominate and fewer
 * splits win.  O(splits x batch x row groups x log SMs) host work.  The plan
 * serves only calls whose lengths are at most the ones given; errors as
 * mla_decode_plan, plus MLA_ERR_INVALID_ARG for a NULL seq_lens or an
 * L_b < q_len.
 */
mla_status_t mla_decode_plan_lengths(int batch, int num_heads, int q_len, const int32_t* seq_lens,
                                     int page_size, mla_kv_dtype_t kv_dtype, int num_sms,
                                     mla_decode_plan_t* plan);

/*
 * mla_workspace_init -- zero the workspace header (the sticky device error
 * word) once after the caller allocates the workspace.  Asynchronous on stream.
 * Library plumbing with no counterpart on the source pages: it exists because
 * the caller, not the library, owns the workspace (the preallocated workspace
 * of the vLLM PR #46819 summary, implementation breakdown 2).
 */
mla_status_t mla_workspace_init(void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * mla_decode -- the whole decode: the split-KV attention kernel, then (when
 * plan->num_kv_splits > 1) the LSE-weighted combine kernel.  The operation is
 * the absorbed-form decode at the top of this header; the call shape (query
 * parts, paged cache, block table, lengths, per-call scales, out + lse) is
 * the TokenSpeed MLA summary's decode interface (vLLM PR #41778,
 * implementation breakdown 1), with the FP8 dequant scale passed on every
 * call as its review highlights ask.
 *
 *   q_nope  : bf16 rows (b,i,h), 512 used, row stride q_nope_row_stride elements
 *   q_pe    : bf16 rows (b,i,h), 64 used, row stride q_pe_row_stride elements
 *             (both strides multiples of 8 elements, base 16-byte aligned)
 *   kv_cache: [num_pages, 64, 576] bf16 or e4m3 bytes (per plan->kv_dtype),
 *             16-byte aligned, rows contiguous
 *   block_table : int32 [batch, block_table_stride]; entries for pages
 *             [0, ceil(L_b/64)) must lie in [0, num_pages); the rest is unread
 *   seq_lens: int32 [batch] on the device, q_len <= L_b <= plan->max_seq_len
 *   softmax_scale : multiplies q.x (1/sqrt(192) for DeepSeek-R1); read per call
 *   kv_scale: device fp32 dequant scale for an FP8 cache (NULL = 1.0); read by
 *             the kernel on every launch, never cached.  With an FP8 cache the
 *             tensor-core operands are f16 (every e4m3 value is exact in f16,
 *             and the conversion is one instruction per pair), so the bf16
 *             query must lie within +-65504: a value beyond that is a
 *             device-side input error (index -4, value = the row i*H + h within
 *             the request) and that row alone is written as NaN
 *   out     : [batch, q_len, H, 512] bf16 or fp32 (out_dtype)
 *   lse     : [batch, q_len, H] fp32 natural-log LSE, or NULL
 *   workspace, workspace_bytes : >= plan->workspace_bytes, 256-byte aligned;
 *             header zeroed once by mla_workspace_init; may be reused by any
 *             later call whose plan needs no more bytes
 *
 * Host-checkable problems return at once, before any launch.  Problems only the
 * device can see (seq_len out of range, a page index outside [0, num_pages),
 * a wait that timed out) set the sticky error word in the workspace header and
 * the affected request's rows are written as NaN; mla_decode_check_error
 * reports them.  Non-uniform q_len goes through mla_decode_varlen; there is
 * no fallback.
 */
mla_status_t mla_decode(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                        const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
                        int num_pages, const int32_t* block_table, int block_table_stride,
                        const int32_t* seq_lens, float softmax_scale, const float* kv_scale,
                        void* out, mla_out_dtype_t out_dtype, float* lse, void* workspace,
                        size_t workspace_bytes, void* cuda_stream);

/*
 * mla_split_kv -- the first stage alone (paged KV gather, QK^T, online
 * softmax with the causal mask, PV, split epilogue); the per-split partial of
 * width kv_lora_rank + 1 follows the attn_logits layout of the vLLM PR #46819
 * summary (key code excerpt).  Same arguments as mla_decode.
 *
 * Request b uses s_b = clamp(ceil(L_b / chunk_tokens), 1, num_kv_splits)
 * splits.  With s_b = 1 the stage writes the request's out/lse directly (and,
 * when the plan has more splits, +inf as the LSE of its first partial, which
 * tells mla_combine to leave those rows alone).  Otherwise it writes fp32
 * partials [B, q_len, H, splits, 513] into the workspace: for splits below s_b
 * the 512 normalised outputs and the split's LSE (-inf if no row of the split
 * sees a token), for the others only an LSE of -inf.
 */
mla_status_t mla_split_kv(const mla_decode_plan_t* plan, const void* q_nope,
                          int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                          const void* kv_cache, int num_pages, const int32_t* block_table,
                          int block_table_stride, const int32_t* seq_lens, float softmax_scale,
                          const float* kv_scale, void* out, mla_out_dtype_t out_dtype, float* lse,
                          void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * mla_combine -- the second stage alone: for every row, M = max_s lse_s,
 * lse = M + ln sum_s exp(lse_s - M), out = sum_s exp(lse_s - lse) * o_s, read
 * from the partials mla_split_kv wrote (the split-KV reduction whose partials
 * carry one LSE per split, vLLM PR #46819 summary, key code excerpt).  A
 * no-op when the plan has one split.
 */
mla_status_t mla_combine(const mla_decode_plan_t* plan, void* out, mla_out_dtype_t out_dtype,
                         float* lse, const void* workspace, size_t workspace_bytes,
                         void* cuda_stream);

/*
 * mla_decode_varlen -- mla_decode with a number of query tokens per request
 * (the per-request metadata the TokenSpeed MLA summary asks for in place of a
 * fallback that unsqueezes non-uniform q_len; vLLM PR #41778, review
 * highlights and risk 6).
 *
 * Same arguments as mla_decode plus
 *   q_lens : int32 [batch] on the device, 1 <= q_lens[b] <= plan->q_len and
 *            q_lens[b] <= seq_lens[b]
 * The layouts stay padded to plan->q_len: request b's query rows are (b, i, h)
 * for i < q_lens[b]; its query i sees tokens [0, L_b - q_lens[b] + i], so each
 * request's last query token sits at position L_b - 1.  Rows with
 * i >= q_lens[b] are padding: their out rows are written as 0 and their lse as
 * -inf, whatever q_nope/q_pe hold there.  A q_lens[b] out of range is a
 * device-side input error (index -2, value q_lens[b]) that writes request b's
 * rows as NaN.  q_lens == NULL returns MLA_ERR_INVALID_ARG.
 */
mla_status_t mla_decode_varlen(const mla_decode_plan_t* plan, const void* q_nope,
                               int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                               const void* kv_cache, int num_pages, const int32_t* block_table,
                               int block_table_stride, const int32_t* seq_lens, const int32_t* q_lens,
                               float softmax_scale, const float* kv_scale, void* out,
                               mla_out_dtype_t out_dtype, float* lse, void* workspace,
                               size_t workspace_bytes, void* cuda_stream);

/*
 * mla_decode_fp8 -- mla_decode with an FP8 query over an FP8 cache, and an
 * optional FP8 output (the TokenSpeed MLA summary: the decode is handed FP8
 * scales, output_scale among them, implementation breakdown 1; its review
 * names the follow-up "pass output_scale and assert FP8 Q").  QK^T runs on
 * the e4m3 codes of query and cache on the FP8 tensor path (products of e4m3
 * codes are exact, so the scores equal those on the dequantised values up to
 * fp32 summation order); P and V stay 16-bit (f16) for PV, V being the cache
 * codes widened exactly.
 *
 * Same arguments as mla_decode, except:
 *   plan    : kv_dtype must be MLA_KV_FP8_E4M3 (else MLA_ERR_UNSUPPORTED)
 *   q_nope, q_pe : e4m3 codes, rows (b,i,h), 512 and 64 used; row strides in
 *             elements (= bytes), multiples of 16; bases 16-byte aligned
 *   q_scale : device fp32, query = code * q_scale (one per-tensor scale for
 *             q_nope and q_pe; NULL = 1.0); read on every launch
 *   out_dtype : MLA_OUT_BF16, MLA_OUT_FP32 or MLA_OUT_FP8_E4M3
 *   out_scale : device fp32 for MLA_OUT_FP8_E4M3 (NULL = 1.0): every output
 *             element is the e4m3 code of out / out_scale, rounded to nearest
 *             even and saturated to +-448 (NaN rows of a rejected request stay
 *             NaN); ignored for the other output types
 * lse stays fp32.
 */
mla_status_t mla_decode_fp8(const mla_decode_plan_t* plan, const void* q_nope, int64_t q_nope_row_stride,
                            const void* q_pe, int64_t q_pe_row_stride, const float* q_scale,
                            const void* kv_cache, int num_pages, const int32_t* block_table,
                            int block_table_stride, const int32_t* seq_lens, float softmax_scale,
                            const float* kv_scale, void* out, mla_out_dtype_t out_dtype,
                            const float* out_scale, float* lse, void* workspace, size_t workspace_bytes,
                            void* cuda_stream);

/*
 * mla_decode_shard -- one rank's part of a decode whose cache is sharded by
 * sequence across ranks (decode context parallelism: each rank holds a
 * contiguous range of every request's tokens and attends over it with all
 * query heads, and the ranks' partial outputs are merged by LSE; the vLLM PR
 * #46819 summary reserves its split partials for num_heads * dcp_world_size
 * query heads in the key code excerpt, and the vLLM PR #47327 report makes
 * its workspace DCP-aware in implementation breakdown 1).
 *
 * Same arguments as mla_decode, except:
 *   kv_cache, block_table : this rank's own paged cache; local token t of
 *             request b is absolute position shard_start[b] + t and lives at
 *             block_table[b, t / 64], slot t % 64
 *   shard_lens  : int32 [batch] on the device, tokens of request b this rank
 *             holds (0 allowed); plan->max_seq_len >= every shard_lens[b]
 *   shard_start : int32 [batch] on the device, absolute position of the
 *             rank's first token of request b
 *   seq_lens    : int32 [batch] on the device, the whole length L_b of request
 *             b (the q_len new tokens included): query i sees absolute
 *             positions [0, L_b - q_len + i], so the mask stays causal
 *   shard_partial : fp32 [batch, q_len, H, 513], 4-byte aligned: per query row
 *             the normalised output over the positions it sees in this shard,
 *             then that part's natural-log LSE (0 and -inf if it sees none)
 * A request with shard_start < 0, shard_start + shard_lens > L_b or
 * L_b < q_len is a device-side input error (index -3 or -1) and its rows are
 * written as NaN.
 */
mla_status_t mla_decode_shard(const mla_decode_plan_t* plan, const void* q_nope,
                              int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                              const void* kv_cache, int num_pages, const int32_t* block_table,
                              int block_table_stride, const int32_t* shard_lens,
                              const int32_t* shard_start, const int32_t* seq_lens, float softmax_scale,
                              const float* kv_scale, float* shard_partial, void* workspace,
                              size_t workspace_bytes, void* cuda_stream);

/*
 * mla_combine_shards -- the LSE merge of the shards' partials (the same merge
 * as mla_combine, over ranks instead of splits).
 *   rows           : batch * q_len * H
 *   shard_partials : fp32 [num_shards, rows, 513], shard-major (what an
 *                    all-gather of every rank's shard_partial produces)
 *   out, lse       : as for mla_decode ([rows, 512] and [rows])
 * Rows whose shards are all empty get out = 0 and lse = -inf; a NaN LSE in any
 * shard (a rejected request) makes the row NaN.
 */
mla_status_t mla_combine_shards(int64_t rows, int num_shards, const float* shard_partials, void* out,
                                mla_out_dtype_t out_dtype, float* lse, void* cuda_stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device
 * memory (code running inside a host framework that owns every device
 * allocation, or a plug-in handed only input/output pointers).  No counterpart
 * exists on the source pages: it is an addition of this library.
 *
 * Same arguments as mla_decode without the workspace: the workspace is a
 * fixed array of MLA_NOALLOC_SCRATCH_BYTES inside the library's device image,
 * reserved on every GPU that loads the library until the process exits.
 * Nothing is allocated by this call.
 *   - plan->workspace_bytes above MLA_NOALLOC_SCRATCH_BYTES returns
 *     MLA_ERR_WORKSPACE_TOO_SMALL before any launch (plan with fewer splits;
 *     one split needs only the 256-byte header).
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents; calls that may overlap on the GPU race on it, so order them.
 *   - The first call on a device looks up and caches the array's device
 *     address; make it before any stream capture starts.  The cached address
 *     belongs to the device's current context: after cudaDeviceReset it is
 *     stale, so do not call this entry point again in that process.
 *   - The error word is cleared at the start of each call and the caller has
 *     no workspace pointer to read it with, so device-side problems show up
 *     only in the outputs: an input error (bad seq_len or page index) and a
 *     bounded wait that ran out (a timeout) both write the affected rows of
 *     out and lse as NaN.  Callers check the outputs for NaN.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
mla_status_t mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q_nope,
                                int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                                const void* kv_cache, int num_pages, const int32_t* block_table,
                                int block_table_stride, const int32_t* seq_lens, float softmax_scale,
                                const float* kv_scale, void* out, mla_out_dtype_t out_dtype, float* lse,
                                void* cuda_stream);

/*
 * mla_decode_check_error -- synchronises the stream, reads the sticky device
 * error word from the workspace header, clears it, and returns MLA_OK,
 * MLA_ERR_DEVICE_INPUT or MLA_ERR_TIMEOUT (or MLA_ERR_CUDA if the stream
 * itself failed).  info (may be NULL) receives {code, request, index, value}.
 * It is how device-side errors surface instead of going unnoticed (the
 * TokenSpeed MLA summary, risks and impact item 6, warns that a leftover
 * fallback path can turn a mismatched batch into an out-of-bounds access).
 */
mla_status_t mla_decode_check_error(void* workspace, void* cuda_stream, int32_t info[4]);

/* Human-readable name of a status code (static storage).  Library plumbing;
 * no passage of the source pages corresponds to it. */
const char* mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
