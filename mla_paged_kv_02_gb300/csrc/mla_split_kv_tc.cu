// mla_split_kv_tc.cu -- split-KV MLA decode attention on the 5th-generation
// tensor cores (tcgen05 + TMEM) with TMA page loads, for sm_103a.
//
// One CTA = (row group of 64 query rows, split, request).  Its split covers
// tokens [split*chunk, min((split+1)*chunk, L)) of request b; every page of it
// is read once from HBM and shared by all 64 rows (the "one KV read per tile
// for all heads and MTP rows" reading of the TokenSpeed MLA summary's
// sub-linear KV scan claim, vLLM PR #41778, motivation).
//
// Warp roles (192 threads):
//   warp 0  TMA producer: Q once (9 boxes of 64 rows x 64 cols), then per page a
//           block_table lookup and 9 boxes of 64 tokens x 64 cols (128B swizzle)
//           into a 2-stage ring; owns the TMEM allocation.
//   warp 1  MMA issuer (one thread):
//             QK^T : S[64 rows x 64 tok] (TMEM) = Q[64 x 576] . K[64 x 576]^T,
//                    tcgen05 kind::f16 M=64 N=64, 36 K-steps, both K-major.
//             PV   : O^T[512 dims x 64 rows] (TMEM) += V^T . P^T, four M=128
//                    dim blocks, N=64, 4 K-steps; V^T is the page's first 512
//                    columns read MN-major, P is K-major.
//   warps 6-9  (FP8 cache only) converter warpgroup: the page arrives as e4m3
//           bytes in the upper half of the stage; every thread first pulls its
//           share into registers, then the group writes exact bf16 values (e4m3 is
//           a subset of bf16) in the 128B-swizzled layout the MMAs read.  The
//           per-tensor scale is folded into the softmax scale and the epilogue.
//   warps 2-5  softmax / correction / epilogue warpgroup.  Lanes 0-15 of each
//           warp own one query row each (the M=64 accumulator places row r in
//           TMEM lane 32*(r/16) + r%16).  Online softmax in the exp2 domain with
//           a lazily updated reference max (rescale O only when a row's max
//           grows by more than 2^8), causal mask, zeroing of V rows past L,
//           P (bf16) written into the page's dead k_pe chunk, epilogue O/l.
//
// Shared memory (1 CTA / SM): Q 72 KB + 2 x 72 KB page stages + barriers.
// TMEM: S double buffer at columns [0,128), O^T at [128, 384).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 64;                       // query rows per CTA
constexpr int kChunks = 9;                      // 64-column chunks in a 576-wide row
constexpr int kChunkBytes = 64 * 128;           // 64 rows x 128 B
constexpr int kStageBytes = kChunks * kChunkBytes;  // one page of bf16 rows: 72 KB
constexpr int kStages = 2;
constexpr int kQOff = 0;
constexpr int kStageOff = kQOff + kChunks * kChunkBytes;
constexpr int kCtlOff = kStageOff + kStages * kStageBytes;
constexpr int kSmemBytes = kCtlOff + 2048 + 1024;  // control block + 1 KB alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // two 64-column S buffers
constexpr uint32_t kColO = 128;   // four 64-column O^T blocks (dims 128b .. 128b+127)

constexpr int kSoftmaxWarp0 = 2;
constexpr int kConvWarp0 = 6;
constexpr int kRawOff = kStageBytes / 2;        // e4m3 page (36 KB) in the upper half of a stage
constexpr int kRawBox = 64 * 64;                // one 64 tokens x 64 bytes box

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far above any legitimate wait
constexpr int kPrefetchPages = 4;  // pages pulled into L2 ahead of the 2-stage shared-memory ring

constexpr uint32_t kIdescQK = idesc_bf16(64, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true, false);

struct Ctl {
  uint64_t q_full;
  uint64_t raw_full[kStages];  // FP8: e4m3 bytes landed
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[kStages];
  uint64_t s_free[kStages];
  uint64_t p_full[kStages];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int poisoned;
  float fac[kRows];
  float inv_l[kRows];
  float lse[kRows];
};
static_assert(sizeof(Ctl) <= 2048, "control block");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier over the softmax warpgroup (barrier 1, 128 threads), with an OR
// reduction of a predicate.
__device__ __forceinline__ bool wg_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void conv_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ bool conv_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 2, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Two e4m3 codes (low byte first) -> two bf16 values, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(Ctl* c, uint64_t* bar, uint32_t parity, const DecodeParams& p,
                                         int where) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(a, parity)) return true;
    if (*(volatile int*)&c->abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *(volatile int*)&c->abort = 1;
      report_error(p.err, MLA_ERR_TIMEOUT, blockIdx.z, where, blockIdx.y);
      return false;
    }
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? 320 : 192, 1)
    split_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                       const __grid_constant__ CUtensorMap tm_kv, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  uint8_t* sQ = smem + kQOff;
  uint8_t* sKV = smem + kStageOff;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rg = blockIdx.x;     // row group
  const int split = blockIdx.y;  // split index
  const int b = blockIdx.z;      // request

  const int L = p.seq_lens[b];
  const bool len_ok = seq_len_ok(p, L);
  const int lo = split * p.chunk_tokens;
  const int hi = len_ok ? min(lo + p.chunk_tokens, L) : lo;
  const int first_page = lo / kPage;
  const int n_pages = hi > lo ? (hi + kPage - 1) / kPage - first_page : 0;
  const int row0 = rg * kRows;  // first row of this group within the request
  const float kv_scale = (kFp8 && p.kv_scale) ? *p.kv_scale : 1.0f;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->raw_full[s], 1);
      mbar_init(&ctl->full[s], kFp8 ? 4 : 1);
      mbar_init(&ctl->empty[s], 1);
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_free[s], 4);
      mbar_init(&ctl->p_full[s], 4);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ctl->poisoned = len_ok ? 0 : 1;
    fence_mbarrier_init();
    if (!len_ok && split == 0 && rg == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, -1, L);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_pages > 0) {
      prefetch_tmap(&tm_kv);
      // A page is one contiguous 64 x 576 block of the cache: pull the next few into
      // L2 so that a stage, once freed, refills at L2 rather than HBM latency.
      const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride + first_page;
      const int64_t page_bytes = (int64_t)kPage * kRow * (kFp8 ? 1 : 2);
      auto prefetch_page = [&](int j) {
        if (j < n_pages) {
          const int pg = bt_row[j];
          if (pg >= 0 && pg < p.num_pages)
            prefetch_l2(static_cast<const uint8_t*>(p.kv) + pg * page_bytes, (uint32_t)page_bytes);
        }
      };
      for (int j = 0; j < kPrefetchPages; ++j) prefetch_page(j);
      const int qrow = b * p.rows + row0;
      mbar_arrive_expect_tx(&ctl->q_full, kChunks * kChunkBytes);
      for (int c = 0; c < 8; ++c) tma_load_2d(sQ + c * kChunkBytes, &tm_qn, &ctl->q_full, c * 64, qrow);
      tma_load_2d(sQ + 8 * kChunkBytes, &tm_qp, &ctl->q_full, 0, qrow);
      int issued = 0;
      for (int j = 0; j < n_pages; ++j) {
        const int s = j & 1;
        if (!wait_bar(ctl, &ctl->empty[s], ((j >> 1) & 1) ^ 1, p, 1)) break;
        prefetch_page(j + kPrefetchPages);
        const int page = bt_row[j];
        uint64_t* land = kFp8 ? &ctl->raw_full[s] : &ctl->full[s];
        if (page < 0 || page >= p.num_pages) {
          report_error(p.err, MLA_ERR_DEVICE_INPUT, b, first_page + j, page);
          mbar_arrive(land);  // nothing to load; consumers mask the whole page
        } else if (kFp8) {
          mbar_arrive_expect_tx(land, kChunks * kRawBox);
          uint8_t* dst = sKV + s * kStageBytes + kRawOff;
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kRawBox, &tm_kv, land, c * 64, page * kPage);
        } else {
          mbar_arrive_expect_tx(land, kStageBytes);
          uint8_t* dst = sKV + s * kStageBytes;
          for (int c = 0; c < kChunks; ++c) tma_load_2d(dst + c * kChunkBytes, &tm_kv, land, c * 64, page * kPage);
        }
        issued = j + 1;
      }
      // Never leave with copies in flight: wait (bounded) for the last stages to land.
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        uint64_t* land = kFp8 ? &ctl->raw_full[j & 1] : &ctl->full[j & 1];
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(land), (j >> 1) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_pages > 0) {
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      const uint64_t q_desc = sdesc_sw128(q_addr, 16, 1024);
      bool ok = wait_bar(ctl, &ctl->q_full, 0, p, 2);
      int pv_issued = 0;
      auto issue_pv = [&](int j) -> bool {
        const int s = j & 1;
        if (!wait_bar(ctl, &ctl->p_full[s], (j >> 1) & 1, p, 5)) return false;
        tc_fence_after();
        const uint32_t st = kv_addr + s * kStageBytes;
        const uint64_t v_desc = sdesc_sw128(st, 8192, 1024);
        const uint64_t p_desc = sdesc_sw128(st + 8 * kChunkBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int blk = 0; blk < 4; ++blk)
            mma_bf16_ss(tmem + kColO + blk * 64, v_desc + (uint64_t)((blk * 2 * kChunkBytes + kk * 2048) >> 4),
                        p_desc + (uint64_t)((kk * 32) >> 4), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&ctl->empty[s]);  // frees the stage and marks O^T current through page j
        ++pv_issued;
        return true;
      };
      for (int j = 0; ok && j < n_pages; ++j) {
        const int s = j & 1;
        if (!wait_bar(ctl, &ctl->full[s], (j >> 1) & 1, p, 3)) { ok = false; break; }
        if (!wait_bar(ctl, &ctl->s_free[s], ((j >> 1) & 1) ^ 1, p, 4)) { ok = false; break; }
        tc_fence_after();
        const uint64_t k_desc = sdesc_sw128(kv_addr + s * kStageBytes, 16, 1024);
        const uint32_t d = tmem + kColS + s * 64;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(d, q_desc + (uint64_t)((c * kChunkBytes + k * 32) >> 4),
                        k_desc + (uint64_t)((c * kChunkBytes + k * 32) >> 4), kIdescQK, (c | k) ? 1u : 0u);
        mma_commit(&ctl->s_full[s]);
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_pages - 1);
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      mma_commit(&ctl->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      (void)pv_issued;
    }
  } else if (kFp8 && warp >= kConvWarp0) {
    // ------------------------------------------------------------ e4m3 -> bf16 converter
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    for (int j = 0; j < n_pages; ++j) {
      const int s = j & 1;
      // Every decision after a bounded wait is made uniform across the group, so no
      // thread can reach a named barrier that another thread has already left.
      if (conv_sync_or(!wait_bar(ctl, &ctl->raw_full[s], (j >> 1) & 1, p, 9))) break;
      uint8_t* stage = sKV + s * kStageBytes;
      // Unit u = (chunk c, token t): 64 e4m3 bytes at raw box c, row t.  Pull all
      // of this thread's units into registers before anyone overwrites the raw half.
      uint4 raw[5][4];
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int u = ct + k * 128;
        if (u < kChunks * 64) {
          const uint4* src = reinterpret_cast<const uint4*>(stage + kRawOff + (u >> 6) * kRawBox + (u & 63) * 64);
#pragma unroll
          for (int q = 0; q < 4; ++q) raw[k][q] = src[q];
        }
      }
      conv_sync();
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int u = ct + k * 128;
        if (u < kChunks * 64) {
          const int c = u >> 6, t = u & 63;
          uint8_t* dst = stage + c * kChunkBytes + t * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 16 bytes in -> 32 bytes (two swizzled 16-byte units) out
            const uint32_t w[4] = {raw[k][q].x, raw[k][q].y, raw[k][q].z, raw[k][q].w};
            uint32_t o[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              o[2 * h] = e4m3x2_to_bf16x2((uint16_t)(w[h] & 0xFFFFu));
              o[2 * h + 1] = e4m3x2_to_bf16x2((uint16_t)(w[h] >> 16));
            }
            const int u0 = 2 * q, u1 = 2 * q + 1;
            *reinterpret_cast<uint4*>(dst + ((u0 ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + ((u1 ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
      fence_proxy_async_smem();
      conv_sync();  // the raw half of this stage is dead for every thread before the next load
      if (lane == 0) mbar_arrive(&ctl->full[s]);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int wg_t = threadIdx.x - kSoftmaxWarp0 * 32;  // 0..127
    const int quad = warp & 3;                          // TMEM lane quadrant this warp may access
    const int r = quad * 16 + lane;                     // query row within the group (lanes 0-15)
    const bool row_thread = lane < 16 && row0 + r < p.rows;
    const int grow_local = row0 + r;                    // row within the request
    const int qi = grow_local / p.num_heads;            // query index i of this row
    const int vis = L - p.q_len + 1 + qi;               // visible tokens for this row
    const float sc2 = p.softmax_scale * kv_scale * kLog2e;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool poisoned = !len_ok;
    bool ok = true;

    for (int j = 0; j < n_pages; ++j) {
      const int s = j & 1;
      const int tok0 = lo + j * kPage;  // first token of page j (lo is page aligned)
      const int page = p.block_table[(int64_t)b * p.bt_stride + first_page + j];
      const bool page_ok = page >= 0 && page < p.num_pages;
      poisoned |= !page_ok;
      // Uniform across the warpgroup (see the converter): a late arrival cannot split it.
      if (wg_sync_or(!wait_bar(ctl, &ctl->s_full[s], (j >> 1) & 1, p, 6))) { ok = false; break; }
      tc_fence_after();
      __syncwarp();
      float sv[64];
      {
        uint32_t raw[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          tmem_ld16(tmem + lane_base + kColS + s * 64 + g * 16, raw);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) sv[g * 16 + k] = __uint_as_float(raw[k]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free[s]);

      // Mask and scale: token tok0+c is visible to this row iff tok0+c < vis.
      const int n_vis = page_ok ? min(max(vis - tok0, 0), kPage) : 0;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float x = (row_thread && c < n_vis) ? sv[c] * sc2 : -INFINITY;
        sv[c] = x;
        mx = fmaxf(mx, x);
      }
      const bool need = row_thread && (mx > m_ref + kRescaleThreshold);
      if (wg_sync_or(need)) {
        float fac = 1.f;
        if (need) {
          fac = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx);
          l_sum *= fac;
          m_ref = mx;
        }
        if (lane < 16) ctl->fac[r] = fac;
        // O^T holds pages < j once PV(j-1) has completed (its commit also covers
        // every earlier MMA); only then may its columns be rescaled.
        bool fail = j > 0 && !wait_bar(ctl, &ctl->empty[(j - 1) & 1], ((j - 1) >> 1) & 1, p, 7);
        fail = wg_sync_or(fail);  // uniform decision; also publishes fac[]
        tc_fence_after();
        if (fail) { ok = false; break; }
        __syncwarp();
        if (j > 0) {
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
              uint32_t v[16];
              const uint32_t ta = tmem + lane_base + kColO + blk * 64 + g * 16;
              tmem_ld16(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * ctl->fac[g * 16 + k]);
              tmem_st16(ta, v);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
      }

      // P = 2^(x - m_ref) as bf16 into the page's k_pe chunk (dead after QK^T),
      // row r, 128B-swizzled K-major: 16-byte unit u of row r sits at u ^ (r & 7).
      uint8_t* stage = sKV + s * kStageBytes;
      if (row_thread) {
        uint8_t* prow = stage + 8 * kChunkBytes + r * 128;
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float x0 = sv[u * 8 + 2 * h], x1 = sv[u * 8 + 2 * h + 1];
            const float p0 = (x0 == -INFINITY) ? 0.f : ex2(x0 - m_ref);
            const float p1 = (x1 == -INFINITY) ? 0.f : ex2(x1 - m_ref);
            part += p0 + p1;
            __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
            w[h] = *reinterpret_cast<uint32_t*>(&pk);
          }
          *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_sum += part;
      }
      // V rows of tokens at or past L (or of a page that was never loaded) may hold
      // anything, NaN included; zero their 512 c_kv columns so 0 * V stays 0.
      const int n_valid = page_ok ? min(L - tok0, kPage) : 0;
      if (n_valid < kPage) {
        const int t = wg_t & 63;
        if (t >= n_valid) {
          const int c0 = (wg_t >> 6) * 4;
#pragma unroll
          for (int c = c0; c < c0 + 4; ++c) {
            uint4* rowp = reinterpret_cast<uint4*>(stage + c * kChunkBytes + t * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) rowp[u] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[s]);
    }

    // ------------------------------------------------------------ epilogue
    if (row_thread) {
      const bool has = l_sum > 0.f;
      ctl->inv_l[r] = has ? kv_scale / l_sum : 0.f;
      ctl->lse[r] = has ? (m_ref + lg2(l_sum)) * kLn2 : -INFINITY;
    }
    if (poisoned) atomicOr(&ctl->poisoned, 1);
    // O^T is final once PV(n-1) has completed.
    bool fail = !ok || (n_pages > 0 && !wait_bar(ctl, &ctl->empty[(n_pages - 1) & 1], ((n_pages - 1) >> 1) & 1, p, 8));
    fail = wg_sync_or(fail);
    tc_fence_after();
    const bool have_o = !fail && n_pages > 0;
    const bool bad = ctl->poisoned != 0 || fail;
    __syncwarp();
    const int rows_here = min(kRows, p.rows - row0);
    const int64_t grow0 = (int64_t)b * p.rows + row0;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int dim = blk * 128 + quad * 32 + lane;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        uint32_t v[16];
        if (have_o) {
          tmem_ld16(tmem + lane_base + kColO + blk * 64 + g * 16, v);
          tmem_ld_wait();
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int rr = g * 16 + k;
          if (rr >= rows_here) continue;
          const float il = ctl->inv_l[rr];
          float o = (have_o && il > 0.f) ? __uint_as_float(v[k]) * il : 0.f;
          if (bad) o = NAN;
          const int64_t grow = grow0 + rr;
          if (p.splits == 1)
            store_out(p, grow, dim, o);
          else
            p.partials[(grow * p.splits + split) * kPartRow + dim] = o;
        }
      }
    }
    if (wg_t < rows_here) {
      const int64_t grow = grow0 + wg_t;
      const float lv = bad ? NAN : ctl->lse[wg_t];
      if (p.splits == 1) {
        if (p.lse) p.lse[grow] = lv;
      } else {
        p.partials[(grow * p.splits + split) * kPartRow + kKvLora] = lv;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeFn>(f);
  }
  return fn;
}

// 2-D tensor map: `rows` rows of `cols` elements, `stride_elems` apart, box 64 x 64.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_elems,
               CUtensorMapDataType dt, uint32_t elem_bytes, CUtensorMapSwizzle swz) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride_elems * elem_bytes};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_split_kv(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap tm_qn, tm_qp, tm_kv;
  const uint64_t q_rows = (uint64_t)p.batch * p.rows;
  const uint64_t kv_rows = (uint64_t)p.num_pages * kPage;
  if (!encode_2d(&tm_qn, p.q_nope, kKvLora, q_rows, p.q_nope_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_qp, p.q_pe, kRope, q_rows, p.q_pe_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const bool ok = p.kv_fp8 ? encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                                       CU_TENSOR_MAP_SWIZZLE_NONE)
                           : encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  const dim3 grid(p.row_groups, p.splits, p.batch);
  if (p.kv_fp8) {
    auto kern = split_kv_tc_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, 320, kSmemBytes, stream>>>(tm_qn, tm_qp, tm_kv, p);
  } else {
    auto kern = split_kv_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, 192, kSmemBytes, stream>>>(tm_qn, tm_qp, tm_kv, p);
  }
  return cudaGetLastError();
}

}  // namespace mla
