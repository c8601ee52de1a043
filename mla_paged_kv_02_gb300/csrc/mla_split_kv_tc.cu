// mla_split_kv_tc.cu -- split-KV MLA decode attention on the 5th-generation
// tensor cores (tcgen05 + TMEM), TMA page loads and a 2-CTA cluster, for sm_103a.
//
// One cluster of two CTAs = (group of 128 query rows, split, request).  Its
// split covers tokens [split*chunk, min((split+1)*chunk, L)) of request b.  Every
// page of the split is read from HBM once and shared by all 128 rows (the
// "one KV read per tile for all heads and MTP rows" reading of the TokenSpeed
// MLA summary's sub-linear KV scan claim, vLLM PR #41778, motivation).
//
// The 576-wide contraction is split between the two CTAs: CTA 0 holds columns
// [0, 256) of Q and of every page, CTA 1 holds [256, 576) (the rest of c_kv and
// k_pe).  That keeps both operands of every MMA at 128 rows:
//   QK^T : S_c[128 rows x 64 tok] = Q[:, cols_c] . K[:, cols_c]^T  (M=128, N=64)
//   PV   : O_c[128 rows x 256]   += P[128 x 64] . V[64 x cols_c(256)] (M=128, N=256)
// where each CTA's 256 V columns are exactly the first four 64-column chunks it
// already holds.  The two partial S_c are summed across the pair through
// distributed shared memory: CTA c owns the softmax of 64 rows (CTA 0 rows 0-63,
// CTA 1 rows 64-127), receives the peer's partial for those rows, computes P,
// and writes its P rows into both CTAs' P buffers.
//
// Warp roles (192 threads; 320 for an FP8 cache):
//   warp 0     TMA producer: Q once, then per page a block-table lookup and the
//              CTA's 4 or 5 64x64 boxes (128B swizzle) into a 4-stage ring; L2
//              prefetch of upcoming pages; owns the TMEM allocation.
//   warp 1     MMA issuer (one thread).
//   warps 2-5  softmax / exchange / epilogue warpgroup.  Warp w reads TMEM lane
//              quadrant w%4 (rows 32*(w%4) .. +31).  Quadrants of rows this CTA
//              owns compute the softmax; the other two send their S partial rows
//              to the peer.  Online softmax in the exp2 domain with a lazily
//              updated reference max: O is rescaled only when a row's max grows
//              by more than 2^8, coordinated across the pair by a per-page flag.
//   warps 6-9  (FP8 cache) converter: the CTA's e4m3 columns land in the upper
//              half of a stage; every thread first pulls its share into
//              registers, then writes exact bf16 values (e4m3 is a subset of
//              bf16) in the swizzled layout.  The per-tensor scale is folded into
//              the softmax scale and the epilogue.
//
// Q's c_kv columns are kept in tensor memory as the A operand of QK^T (read every
// page; from TMEM they cost no shared-memory bandwidth and leave room for 4 page
// stages); CTA 1's q_pe chunk stays in shared memory.
// TMEM: O_c at columns [0,256), S double buffer at [256,384), Q at [384,512).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 128;              // query rows per cluster
constexpr int kMaxCh = 5;               // 64-column chunks a CTA holds (CTA 0: 4, CTA 1: 5)
constexpr int kQChunkBytes = 128 * 128;  // 128 rows x 128 B
constexpr int kKvChunkBytes = 64 * 128;  // 64 tokens x 128 B
constexpr int kStageBytes = kMaxCh * kKvChunkBytes;
constexpr int kStages = 4;
constexpr int kSinBytes = 64 * 64 * 4;  // peer's partial S for the 64 owned rows
constexpr int kPBytes = kRows * 128;    // P[128 rows x 64 tokens] bf16
constexpr int kStageOff = 0;
constexpr int kQStageOff = kStageOff + 2 * kStageBytes;  // Q's c_kv chunks land in stages 2-3, then go to TMEM
static_assert(4 * kQChunkBytes <= 2 * kStageBytes, "Q staging");
constexpr int kSinOff = kStageOff + kStages * kStageBytes;  // one S_in buffer
constexpr int kPOff = kSinOff + kSinBytes;                    // two P buffers
constexpr int kQpeOff = kPOff + 2 * kPBytes;                  // CTA 1's q_pe chunk (A from shared memory)
constexpr int kCtlOff = kQpeOff + kQChunkBytes;
constexpr int kCtlBytes = 2048;
constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kPOff % 1024 == 0 && kStageOff % 1024 == 0 && kQpeOff % 1024 == 0, "swizzle atoms");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O_c: 256 columns
constexpr uint32_t kColS = 256;  // S: two 64-column buffers
constexpr uint32_t kColQ = 384;  // Q's c_kv chunks as the A operand: 2 bf16 per column, 128 columns

constexpr int kSoftmaxWarp0 = 2;
constexpr int kConvWarp0 = 6;
constexpr int kRawOff = kStageBytes / 2;  // e4m3 columns of a page in the upper half of a stage
constexpr int kRawBox = 64 * 64;          // one 64 tokens x 64 bytes box

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far above any legitimate wait
constexpr int kPrefetchPages = 4;

constexpr uint32_t kIdescQK = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);

// Per page and owner warp: each row's O rescale factor and whether any row of
// the warp moved its reference max (flag = page + 1).  Copied to the peer with
// the warp's 32 P rows.
struct alignas(16) Meta {
  float fac[32];
  int flag;
  int pad[3];
};
constexpr int kMetaBytes = sizeof(Meta);
constexpr uint32_t kPvReadyTx = 2 * (32 * 128 + kMetaBytes);  // the peer's 2 owner warps' copies

struct Ctl {
  uint64_t q_full;
  uint64_t raw_full[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];     // this CTA's PV of the stage's page has completed
  uint64_t q_tmem;             // Q moved from shared to tensor memory (count 4)
  uint64_t s_full[2];          // QK^T of the page is in TMEM
  uint64_t s_free[2];          // the 4 softmax warps have read it (count 4)
  uint64_t sin_full;           // peer's partial S landed (count 1 + 16 KB of st.async bytes)
  uint64_t sin_free;           // peer's 2 owner warps consumed what this CTA sent (count 2, remote)
  uint64_t p_free[2];          // PV of the buffer's previous page done in both CTAs (count 2)
  uint64_t pv_ready[2];        // local owners wrote P (count 2) + the peer's P and meta copies landed
  uint64_t rescaled[2];        // the 4 local warps rescaled O (count 4)
  uint64_t fin;                // 1/l of all 128 rows delivered (count 4)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int poisoned;
  Meta meta_local[2][2];       // [page buffer][owner warp]: written by this CTA's owners
  Meta meta_peer[2][2];        // the same, copied in from the peer
  float inv_l[kRows];
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

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

// Named barrier over the softmax warpgroup (barrier 1, 128 threads), OR-reducing
// a predicate.  Every decision that follows a bounded wait goes through it, so
// no thread can reach a later barrier that another thread has already left.
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

// Bounded wait that also gives up once any role of this CTA has aborted.  CTA
// scope suffices for every barrier completed by local arrives, by transaction
// bytes (TMA, st.async, bulk copies) or by a relaxed "consumed" signal; only a
// barrier whose remote arrivals publish generic stores needs cluster scope.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(Ctl* c, uint64_t* bar, uint32_t parity, const DecodeParams& p,
                                         int where) {
  const uint32_t a = smem_u32(bar);
  auto test = [&]() { return kCluster ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity); };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (test()) return true;
    if (*(volatile int*)&c->abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *(volatile int*)&c->abort = 1;
      report_error(p.err, MLA_ERR_TIMEOUT, blockIdx.z, where, blockIdx.y);
      return false;
    }
  }
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFp8 ? 320 : 192, 1)
    split_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                       const __grid_constant__ CUtensorMap tm_kv, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  uint8_t* sQ = smem + kQStageOff;  // Q staging (then stages 2-3)
  uint8_t* sKV = smem + kStageOff;
  uint8_t* sSin = smem + kSinOff;
  uint8_t* sQpe = smem + kQpeOff;
  uint8_t* sP = smem + kPOff;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();  // 0 or 1: which column half this CTA holds
  const uint32_t peer = cta ^ 1u;
  const int nch = cta == 0 ? 4 : 5;        // 64-column chunks held
  const int g0 = cta == 0 ? 0 : 4;         // first global chunk
  const int rg = blockIdx.x >> 1;          // row group
  const int split = blockIdx.y;
  const int b = blockIdx.z;

  const int L = p.seq_lens[b];
  const bool len_ok = seq_len_ok(p, L);
  const int lo = split * p.chunk_tokens;
  const int hi = len_ok ? min(lo + p.chunk_tokens, L) : lo;
  const int first_page = lo / kPage;
  const int n_pages = hi > lo ? (hi + kPage - 1) / kPage - first_page : 0;
  const int row0 = rg * kRows;
  const float kv_scale = (kFp8 && p.kv_scale) ? *p.kv_scale : 1.0f;
  const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride + first_page;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->raw_full[s], 1);
      mbar_init(&ctl->full[s], kFp8 ? 4 : 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->q_tmem, 4);
    mbar_init(&ctl->s_full[0], 1);
    mbar_init(&ctl->s_full[1], 1);
    mbar_init(&ctl->s_free[0], 4);
    mbar_init(&ctl->s_free[1], 4);
    mbar_init(&ctl->sin_full, 1);
    mbar_init(&ctl->sin_free, 2);
    for (int e = 0; e < 2; ++e) {
      mbar_init(&ctl->p_free[e], 2);
      mbar_init(&ctl->pv_ready[e], 2);
      mbar_init(&ctl->rescaled[e], 4);
      for (int w = 0; w < 2; ++w) ctl->meta_local[e][w].flag = ctl->meta_peer[e][w].flag = 0;
    }
    mbar_init(&ctl->fin, 4);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ctl->poisoned = len_ok ? 0 : 1;
    fence_mbarrier_init();
    if (!len_ok && split == 0 && rg == 0 && cta == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, -1, L);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_pages > 0) {
      prefetch_tmap(&tm_kv);
      const int64_t page_bytes = (int64_t)kPage * kRow * (kFp8 ? 1 : 2);
      // A page is one contiguous block of the cache; CTA 0 pulls the next few
      // whole pages into L2 so that freed stages refill at L2 latency.
      auto prefetch_page = [&](int j) {
        if (cta == 0 && j < n_pages) {
          const int pg = bt_row[j];
          if (pg >= 0 && pg < p.num_pages)
            prefetch_l2(static_cast<const uint8_t*>(p.kv) + pg * page_bytes, (uint32_t)page_bytes);
        }
      };
      for (int j = 0; j < kPrefetchPages; ++j) prefetch_page(j);
      const int qrow = b * p.rows + row0;
      mbar_arrive_expect_tx(&ctl->q_full, nch * kQChunkBytes);
      for (int k = 0; k < nch; ++k) {
        const int g = g0 + k;
        if (g < 8)
          tma_load_2d(sQ + k * kQChunkBytes, &tm_qn, &ctl->q_full, g * 64, qrow);
        else
          tma_load_2d(sQpe, &tm_qp, &ctl->q_full, 0, qrow);
      }
      int issued = 0;
      int next_page = bt_row[0];
      for (int j = 0; j < n_pages; ++j) {
        const int s = j & 3;
        const int page = next_page;
        if (j + 1 < n_pages) next_page = bt_row[j + 1];  // lookups ahead of the waits
        const int pf = (cta == 0 && j + kPrefetchPages < n_pages) ? bt_row[j + kPrefetchPages] : -1;
        // Stages 2-3 hold Q until the softmax warps have moved it into TMEM.
        if (j == 2 && !wait_bar(ctl, &ctl->q_tmem, 0, p, 17)) break;
        if (!wait_bar(ctl, &ctl->empty[s], ((j >> 2) & 1) ^ 1, p, 1)) break;
        if (pf >= 0 && pf < p.num_pages)
          prefetch_l2(static_cast<const uint8_t*>(p.kv) + pf * page_bytes, (uint32_t)page_bytes);
        uint64_t* land = kFp8 ? &ctl->raw_full[s] : &ctl->full[s];
        uint8_t* stage = sKV + s * kStageBytes;
        if (page < 0 || page >= p.num_pages) {
          if (cta == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, first_page + j, page);
          mbar_arrive(land);  // nothing to load; consumers mask the whole page
        } else if (kFp8) {
          mbar_arrive_expect_tx(land, nch * kRawBox);
          for (int k = 0; k < nch; ++k)
            tma_load_2d(stage + kRawOff + k * kRawBox, &tm_kv, land, (g0 + k) * 64, page * kPage);
        } else {
          mbar_arrive_expect_tx(land, nch * kKvChunkBytes);
          for (int k = 0; k < nch; ++k)
            tma_load_2d(stage + k * kKvChunkBytes, &tm_kv, land, (g0 + k) * 64, page * kPage);
        }
        issued = j + 1;
      }
      // Never leave with copies in flight.
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        uint64_t* land = kFp8 ? &ctl->raw_full[j & 3] : &ctl->full[j & 3];
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(land), (j >> 2) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_pages > 0) {
      const uint32_t kv_addr = smem_u32(sKV);
      const uint32_t p_addr = smem_u32(sP);
      const uint64_t qpe_desc = sdesc_sw128(smem_u32(sQpe), 16, 1024);
      int nres[2] = {0, 0};
      bool ok = wait_bar(ctl, &ctl->q_tmem, 0, p, 2);
      // Greedy issue: QK(nq) as soon as its page has landed and S is free, PV(np)
      // as soon as both CTAs' P(np) is in (and O rescaled, if flagged).  Polling
      // with non-blocking tests keeps one pending PV from holding back the next
      // page's QK.  The stage ring, S, S_in and P barriers bound how far QK runs
      // ahead.
      int nq = 0, np = 0;
      int resc_state = 0;  // for page np: 0 = flags not read, 1 = no rescale, 2 = waiting for rescale
      uint64_t t_last = globaltimer_ns();
      while (ok && np < n_pages) {
        bool progressed = false;
        if (nq < n_pages && mbar_test_wait(smem_u32(&ctl->full[nq & 3]), (nq >> 2) & 1) &&
            mbar_test_wait(smem_u32(&ctl->s_free[nq & 1]), ((nq >> 1) & 1) ^ 1)) {
          tc_fence_after();
          const uint64_t k_desc = sdesc_sw128(kv_addr + (nq & 3) * kStageBytes, 16, 1024);
          const uint32_t d = tmem + kColS + (nq & 1) * 64;
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // A = Q chunk k from TMEM: 16 k per MMA = 8 columns
              mma_bf16_ts(d, tmem + kColQ + k * 32 + kk * 8,
                          k_desc + (uint64_t)((k * kKvChunkBytes + kk * 32) >> 4), kIdescQK, (k | kk) ? 1u : 0u);
          }
          if (nch == 5) {  // k_pe: A = q_pe from shared memory
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss(d, qpe_desc + (uint64_t)((kk * 32) >> 4),
                          k_desc + (uint64_t)((4 * kKvChunkBytes + kk * 32) >> 4), kIdescQK, 1u);
          }
          mma_commit(&ctl->s_full[nq & 1]);
          ++nq;
          progressed = true;
        }
        if (np < nq) {
          const int e = np & 1;
          if (resc_state == 0 && mbar_test_wait(smem_u32(&ctl->pv_ready[e]), (np >> 1) & 1)) {
            const volatile Meta* ml = ctl->meta_local[e];
            const volatile Meta* mp = ctl->meta_peer[e];
            resc_state = (ml[0].flag == np + 1 || ml[1].flag == np + 1 || mp[0].flag == np + 1 ||
                          mp[1].flag == np + 1) ? 2 : 1;  // some row's reference max moved
          }
          if (resc_state == 2 && mbar_test_wait(smem_u32(&ctl->rescaled[e]), nres[e] & 1)) {
            ++nres[e];
            resc_state = 1;
          }
          if (resc_state == 1) {
            tc_fence_after();
            const uint64_t v_desc = sdesc_sw128(kv_addr + (np & 3) * kStageBytes, kKvChunkBytes, 1024);
            const uint64_t p_desc = sdesc_sw128(p_addr + e * kPBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss(tmem + kColO, p_desc + (uint64_t)((kk * 32) >> 4), v_desc + (uint64_t)((kk * 2048) >> 4),
                          kIdescPV, (np > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&ctl->empty[np & 3]);           // stage free; O current through page np
            mma_commit_multicast(&ctl->p_free[e], 3);  // P buffer e reusable, in both CTAs
            ++np;
            resc_state = 0;
            progressed = true;
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else if (*(volatile int*)&ctl->abort) {
          ok = false;
        } else if (globaltimer_ns() - t_last > kWaitLimitNs) {
          *(volatile int*)&ctl->abort = 1;
          report_error(p.err, MLA_ERR_TIMEOUT, blockIdx.z, 3, blockIdx.y);
          ok = false;
        }
      }
      mma_commit(&ctl->drain);  // every MMA of this thread has completed before TMEM is freed
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  } else if (kFp8 && warp >= kConvWarp0) {
    // ------------------------------------------------------------ e4m3 -> bf16 converter
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    const int units = nch * 64;                    // (chunk, token) pairs of 64 bytes
    for (int j = 0; j < n_pages; ++j) {
      const int s = j & 3;
      if (conv_sync_or(!wait_bar(ctl, &ctl->raw_full[s], (j >> 2) & 1, p, 9))) break;
      uint8_t* stage = sKV + s * kStageBytes;
      uint4 raw[3][4];
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int u = ct + k * 128;
        if (u < units) {
          const uint4* src = reinterpret_cast<const uint4*>(stage + kRawOff + (u >> 6) * kRawBox + (u & 63) * 64);
#pragma unroll
          for (int q = 0; q < 4; ++q) raw[k][q] = src[q];
        }
      }
      conv_sync();  // every raw byte is in registers before the bf16 writes overlap them
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int u = ct + k * 128;
        if (u < units) {
          const int c = u >> 6, t = u & 63;
          uint8_t* dst = stage + c * kKvChunkBytes + t * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t w[4] = {raw[k][q].x, raw[k][q].y, raw[k][q].z, raw[k][q].w};
            uint32_t o[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              o[2 * h] = e4m3x2_to_bf16x2((uint16_t)(w[h] & 0xFFFFu));
              o[2 * h + 1] = e4m3x2_to_bf16x2((uint16_t)(w[h] >> 16));
            }
            *reinterpret_cast<uint4*>(dst + (((2 * q) ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + (((2 * q + 1) ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
      fence_proxy_async_smem();
      conv_sync();
      if (lane == 0) mbar_arrive(&ctl->full[s]);
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ------------------------------------------------------------ softmax / exchange warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // row within the group (TMEM lane)
    const bool owner = (quad >> 1) == (int)cta;  // CTA 0 owns rows 0-63, CTA 1 rows 64-127
    const int ri = r & 63;                       // row index within the owned / sent half
    const bool row_ok = row0 + r < p.rows;
    const int qi = (row0 + r) / p.num_heads;
    const int vis = L - p.q_len + 1 + qi;        // tokens this row may see
    const float sc2 = p.softmax_scale * kv_scale * kLog2e;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t sin_local = smem_u32(sSin);
    const uint32_t sin_peer = mapa_shared(sin_local, peer);
    const uint32_t p_peer = mapa_shared(smem_u32(sP), peer);
    const int ow = quad & 1;  // owner-warp index of this quadrant (CTA 0: quads 0,1; CTA 1: quads 2,3)
    float m_ref = -INFINITY, l_sum = 0.f;
    bool poisoned = !len_ok;
    bool ok = true;

    // Every warp runs this loop on its own: decisions after a bounded wait are
    // made warp-uniform (__all_sync), and no named barrier sits inside the loop,
    // so sender warps run a page ahead of the owners and a warp that gives up
    // cannot strand the others on a barrier.
    //
    // Rescale check for page jj, run at the start of iteration jj+2 (by then both
    // CTAs' P(jj) has long been written, so the wait is free): if any row of either
    // CTA moved its reference max on page jj, each warp rescales its lanes (rows)
    // of O by fac before PV(jj) is issued.  It precedes the wait for S(jj+2):
    // PV(jj) is issued before QK(jj+2), so waiting for S first could deadlock.
    auto rescale_check = [&](int jj) -> bool {
      const int e = jj & 1;
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->pv_ready[e], (jj >> 1) & 1, p, 11))) return false;
      const volatile Meta* ml = ctl->meta_local[e];
      const volatile Meta* mp = ctl->meta_peer[e];
      const bool resc = ml[0].flag == jj + 1 || ml[1].flag == jj + 1 || mp[0].flag == jj + 1 || mp[1].flag == jj + 1;
      if (!resc) return true;
      // O holds pages < jj once PV(jj-1) has completed (its commit covers all before).
      if (jj > 0 &&
          !__all_sync(0xffffffffu, wait_bar(ctl, &ctl->empty[(jj - 1) & 3], ((jj - 1) >> 2) & 1, p, 12)))
        return false;
      tc_fence_after();
      __syncwarp();
      const float f = owner ? ctl->meta_local[e][ow].fac[lane] : ctl->meta_peer[e][ow].fac[lane];
#pragma unroll 1
      for (int g = 0; g < 16; ++g) {
        uint32_t v[16];
        const uint32_t ta = tmem + lane_base + kColO + g * 16;
        tmem_ld16(ta, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
        tmem_st16(ta, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->rescaled[e]);
      return true;
    };

    // Q_c rows into tensor memory: thread = row = TMEM lane; the 128B-swizzled
    // staging rows are un-swizzled into 2-bf16 columns, 32 columns per chunk.
    if (n_pages > 0) {
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->q_full, 0, p, 18))) {
        ok = false;
      } else {
        for (int k = 0; k < 4; ++k) {
          const uint8_t* qrow = sQ + k * kQChunkBytes + r * 128;
          uint32_t w[2][16];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((u ^ (r & 7)) << 4));
            w[u >> 2][(u & 3) * 4 + 0] = v.x;
            w[u >> 2][(u & 3) * 4 + 1] = v.y;
            w[u >> 2][(u & 3) * 4 + 2] = v.z;
            w[u >> 2][(u & 3) * 4 + 3] = v.w;
          }
          tmem_st16(tmem + lane_base + kColQ + k * 32, w[0]);
          tmem_st16(tmem + lane_base + kColQ + k * 32 + 16, w[1]);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->q_tmem);
    }

    // Block-table entries are loaded one page ahead: a global load consumed in
    // the same iteration would stall every page for a full memory latency.
    int page_next = (n_pages > 0 && owner) ? bt_row[0] : 0;
    for (int j = 0; ok && j < n_pages; ++j) {
      const int s = j & 1;   // exchange buffers (S_in, P, meta)
      const int st = j & 3;  // page stage
      const int tok0 = lo + j * kPage;  // lo is page aligned
      const int page = page_next;
      if (owner && j + 1 < n_pages) page_next = bt_row[j + 1];
      const bool page_ok = !owner || (page >= 0 && page < p.num_pages);  // only owners use it
      poisoned |= !page_ok;
      if (j >= 2 && !rescale_check(j - 2)) { ok = false; break; }
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->s_full[s], (j >> 1) & 1, p, 6))) { ok = false; break; }
      tc_fence_after();
      float sv[64];
      {
        uint32_t raw[4][16];
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_ld16(tmem + lane_base + kColS + s * 64 + g * 16, raw[g]);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int k = 0; k < 16; ++k) sv[g * 16 + k] = __uint_as_float(raw[g][k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free[s]);

      if (!owner) {
        // ---- sender: partial S of a row the peer owns -> peer's S_in[s][ri]
        if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->sin_free, (j & 1) ^ 1, p, 13))) {
          ok = false;
          break;
        }
        const uint32_t dst = sin_peer + ri * 256;
        const uint32_t bar = mapa_shared(smem_u32(&ctl->sin_full), peer);
#pragma unroll
        for (int u = 0; u < 16; ++u)
          st_async_v4(dst + ((u ^ (ri & 7)) << 4),
                      make_uint4(__float_as_uint(sv[4 * u]), __float_as_uint(sv[4 * u + 1]),
                                 __float_as_uint(sv[4 * u + 2]), __float_as_uint(sv[4 * u + 3])),
                      bar);
      } else {
        // ---- owner: add the peer's partial, softmax, P into both CTAs
        // The peer's two sender warps deliver 16 KB of st.async bytes per page.
        if (ow == 0 && lane == 0) mbar_arrive_expect_tx(&ctl->sin_full, kSinBytes);
        if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->sin_full, j & 1, p, 14))) {
          ok = false;
          break;
        }
        // Full score = own partial + the peer's partial.  Pages that every row of
        // the warp sees in full (all but a split's last page, normally) take a
        // fast path: add and max on raw scores (the scale is positive, so max
        // commutes with it), then p = 2^(s*scale - m) in one FMA + ex2.  Other
        // pages mask and scale first; masked columns, possibly NaN garbage, become
        // -inf and then exactly 0.
        const float4* src = reinterpret_cast<const float4*>(sSin + ri * 256);
        const int n_vis = (page_ok && row_ok) ? min(max(vis - tok0, 0), kPage) : 0;
        const bool fast = __all_sync(0xffffffffu, n_vis == kPage);
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (fast) {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float4 v = src[u ^ (ri & 7)];
            sv[4 * u] += v.x;
            sv[4 * u + 1] += v.y;
            sv[4 * u + 2] += v.z;
            sv[4 * u + 3] += v.w;
#pragma unroll
            for (int k = 0; k < 4; ++k) mq[k] = fmaxf(mq[k], sv[4 * u + k]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float4 v = src[u ^ (ri & 7)];
            const float a[4] = {sv[4 * u] + v.x, sv[4 * u + 1] + v.y, sv[4 * u + 2] + v.z, sv[4 * u + 3] + v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x = (4 * u + k < n_vis) ? a[k] * sc2 : -INFINITY;
              sv[4 * u + k] = x;
              mq[k] = fmaxf(mq[k], x);
            }
          }
        }
        float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        if (fast) mx *= sc2;
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&ctl->sin_free), peer));

        // V rows of tokens at or past L (or of a page that was never loaded) may
        // hold anything, NaN included; zero this CTA's 256 V columns of them.
        const int n_valid = page_ok ? min(L - tok0, kPage) : 0;
        if (ri >= n_valid) {
          uint8_t* stage = sKV + st * kStageBytes;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4* rowp = reinterpret_cast<uint4*>(stage + c * kKvChunkBytes + ri * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) rowp[u] = make_uint4(0, 0, 0, 0);
          }
        }

        const bool need = row_ok && (mx > m_ref + kRescaleThreshold);
        float fac = 1.f;
        if (need) {
          fac = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx);
          l_sum *= fac;
          m_ref = mx;
        }
        uint4 pk[8];
        float part[4] = {0.f, 0.f, 0.f, 0.f};
        if (fast) {
          const float nm = -m_ref;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float p0 = ex2(fmaf(sv[u * 8 + 2 * h], sc2, nm));
              const float p1 = ex2(fmaf(sv[u * 8 + 2 * h + 1], sc2, nm));
              part[h] += p0 + p1;
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            pk[u] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float x0 = sv[u * 8 + 2 * h], x1 = sv[u * 8 + 2 * h + 1];
              const float p0 = (x0 == -INFINITY) ? 0.f : ex2(x0 - m_ref);
              const float p1 = (x1 == -INFINITY) ? 0.f : ex2(x1 - m_ref);
              part[h] += p0 + p1;
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            pk[u] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        l_sum += (part[0] + part[1]) + (part[2] + part[3]);
        // Both CTAs' PV of page j-2 must be done before P buffer s is rewritten.
        if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->p_free[s], ((j >> 1) & 1) ^ 1, p, 15))) {
          ok = false;
          break;
        }
        const uint32_t off = s * kPBytes + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(sP + off + ((u ^ (r & 7)) << 4)) = pk[u];
        Meta& me = ctl->meta_local[s][ow];
        me.fac[lane] = fac;
        const bool any_need = __any_sync(0xffffffffu, need) && j > 0;  // page 0's PV overwrites O
        if (lane == 0) me.flag = any_need ? j + 1 : 0;
        fence_proxy_async_smem();  // P rows and meta visible to the MMA and the bulk copy engine
        __syncwarp();
        if (lane == 0) {
          // This warp's 32 P rows (4 KB, contiguous) and its meta go to the peer
          // through the async proxy; the peer's pv_ready counts the bytes.
          const uint32_t bar = mapa_shared(smem_u32(&ctl->pv_ready[s]), peer);
          const uint32_t rows_off = s * kPBytes + quad * 32 * 128;
          bulk_copy_to_peer(p_peer + rows_off, sP + rows_off, 32 * 128, bar);
          bulk_copy_to_peer(mapa_shared(smem_u32(&ctl->meta_peer[s][ow]), peer), &me, kMetaBytes, bar);
          if (ow == 0)
            mbar_arrive_expect_tx(&ctl->pv_ready[s], kPvReadyTx);
          else
            mbar_arrive(&ctl->pv_ready[s]);
        }
      }
    }
    if (ok && n_pages >= 2 && !rescale_check(n_pages - 2)) ok = false;
    if (ok && n_pages >= 1 && !rescale_check(n_pages - 1)) ok = false;
    ok = !wg_sync_or(!ok);  // the epilogue decides as one group

    // ------------------------------------------------------------ epilogue
    if (owner) {
      const bool has = l_sum > 0.f;
      const float il = has ? kv_scale / l_sum : 0.f;
      ctl->inv_l[r] = il;
      st_cluster_u32(mapa_shared(smem_u32(&ctl->inv_l[r]), peer), __float_as_uint(il));
      const int64_t grow = (int64_t)b * p.rows + row0 + r;
      if (row_ok) {
        float lv = has ? (m_ref + lg2(l_sum)) * kLn2 : -INFINITY;
        if (poisoned || !ok) lv = NAN;
        if (p.splits == 1) {
          if (p.lse) p.lse[grow] = lv;
        } else {
          p.partials[(grow * p.splits + split) * kPartRow + kKvLora] = lv;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->fin), cta));
        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->fin), peer));
      }
    }
    if (poisoned) atomicOr(&ctl->poisoned, 1);
    bool fail = !wait_bar<true>(ctl, &ctl->fin, 0, p, 16);
    fail |= !ok || (n_pages > 0 && !wait_bar(ctl, &ctl->empty[(n_pages - 1) & 3], ((n_pages - 1) >> 2) & 1, p, 8));
    fail = wg_sync_or(fail);
    tc_fence_after();
    __syncwarp();
    const bool have_o = !fail && n_pages > 0;
    const bool bad = ctl->poisoned != 0 || fail;
    const int rows_here = min(kRows, p.rows - row0);
    const int64_t grow0 = (int64_t)b * p.rows + row0;
    // O_c rows are TMEM lanes: stage 32 rows x 32 columns through shared memory
    // (the P buffers, idle once the last PV has completed) so global stores run
    // along the 512 columns.
    float* tile = reinterpret_cast<float*>(sP) + (warp - kSoftmaxWarp0) * (32 * 33);
    const float il = ctl->inv_l[r];
#pragma unroll 1
    for (int c0 = 0; c0 < 256; c0 += 32) {
      uint32_t v[2][16];
      if (have_o) {
        tmem_ld16(tmem + lane_base + kColO + c0, v[0]);
        tmem_ld16(tmem + lane_base + kColO + c0 + 16, v[1]);
        tmem_ld_wait();
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        float o = (have_o && il > 0.f) ? __uint_as_float(v[k >> 4][k & 15]) * il : 0.f;
        if (bad) o = NAN;
        tile[lane * 33 + k] = o;
      }
      __syncwarp();
      const int dim = (int)cta * 256 + c0 + lane;
#pragma unroll 4
      for (int rr = 0; rr < 32; ++rr) {
        const int row = quad * 32 + rr;
        if (row >= rows_here) break;
        const float o = tile[rr * 33 + lane];
        const int64_t grow = grow0 + row;
        if (p.splits == 1)
          store_out(p, grow, dim, o);
        else
          p.partials[(grow * p.splits + split) * kPartRow + dim] = o;
      }
      __syncwarp();
    }
    tc_fence_before();
  }

  __syncthreads();
  cluster_sync_all();  // no remote store or arrive can target a CTA that has exited
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

// 2-D tensor map: `rows` rows of `cols` elements, `stride_elems` apart, box 64 x box_rows.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_elems,
               CUtensorMapDataType dt, uint32_t elem_bytes, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride_elems * elem_bytes};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_split_kv(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap tm_qn, tm_qp, tm_kv;
  const uint64_t q_rows = (uint64_t)p.batch * p.rows;
  const uint64_t kv_rows = (uint64_t)p.num_pages * kPage;
  if (!encode_2d(&tm_qn, p.q_nope, kKvLora, q_rows, p.q_nope_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_qp, p.q_pe, kRope, q_rows, p.q_pe_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const bool ok = p.kv_fp8 ? encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64,
                                       CU_TENSOR_MAP_SWIZZLE_NONE)
                           : encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  const dim3 grid(2 * p.row_groups, p.splits, p.batch);
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
