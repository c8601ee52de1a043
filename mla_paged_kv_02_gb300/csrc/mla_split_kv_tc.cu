// mla_split_kv_tc.cu -- split-KV MLA decode attention on the 5th-generation
// tensor cores (tcgen05 + TMEM), TMA page loads and a 2-CTA cluster, for sm_103a.
//
// One cluster of two CTAs = (group of 128 query rows, split, request).  Its
// split covers tokens [split*chunk, min((split+1)*chunk, L)) of request b.  Every
// page of the split is read from HBM once and shared by all 128 rows (the
// "one KV read per tile for all heads and MTP rows" reading of the TokenSpeed
// MLA summary's sub-linear KV scan claim, vLLM PR #41778, motivation).
//
// The 576-wide contraction is split between the two CTAs: CTA c holds c_kv
// columns [256c, 256c+256) and k_pe columns [32c, 32c+32) of Q and of every
// page.  That keeps both operands of every MMA at 128 rows:
//   QK^T : S_c[128 rows x 64 tok] = Q[:, cols_c] . K[:, cols_c]^T  (M=128, N=64)
//   PV   : O_c[128 rows x 256]   += P[128 x 64] . V[64 x cols_c(256)] (M=128, N=256)
// where each CTA's 256 V columns are exactly the first four 64-column chunks it
// already holds.  The two partial S_c are summed across the pair through
// distributed shared memory, split by tokens: CTA c owns the softmax of tokens
// [32c, 32c+32) of every page for all 128 rows, receives the peer's partial for
// that half, computes P for it, and writes it into both CTAs' P buffers.  The
// bulk transfers between the pair (partial scores, P halves) are bulk copies,
// which the copy engine carries while the warps go on; the per-row reference
// maxima and row sums go by st.async.  Both complete transaction bytes on the
// receiver's mbarrier.
//
// Warp roles (352 threads; 480 with an FP8 cache):
//   warp 0     TMA producer: Q once, then per page a block-table lookup and the
//              CTA's columns of the page into a 4-stage ring (bf16: one 3-D box
//              of four 64x64 chunks, 128B swizzle, and one 32-column k_pe box,
//              64B swizzle; FP8: two 128B-swizzled boxes of 128 e4m3 codes and
//              one 32B-swizzled box of 32); owns the TMEM allocation.
//   warp 1     QK^T issuer (one thread).
//   warps 2-5  softmax / exchange / epilogue warpgroup.  Warp w reads TMEM lane
//              quadrant w%4 (rows 32*(w%4) .. +31) and works on its CTA's token
//              half of those rows.  Online softmax in the exp2 domain with lazily
//              raised whole-number reference maxima, agreed between the pair one
//              page behind (see the warpgroup's comment).
//   warps 6-9  (bf16 cache; 10-13 with an FP8 cache) S senders: the peer's
//              token half of S(j) from TMEM to the peer, off the softmax warps'
//              chain.
//   warps 6-9  (FP8 cache) converter: the CTA's e4m3 columns land at stage +
//              16 KB; each thread pulls one token row of codes into registers,
//              then writes exact f16 values (every e4m3 value is an f16) in the
//              swizzled layout.  The per-tensor scale is folded into the softmax
//              scale and the epilogue.
//   warp 10    PV issuer (one thread; warp 14 with an FP8 cache).
//
// Q's c_kv columns are kept in tensor memory as the A operand of QK^T (read every
// page; from TMEM they cost no shared-memory bandwidth and leave room for 4 page
// stages); the CTA's q_pe columns stay in shared memory.
// TMEM: O_c at columns [0,256), S double buffer at [256,384), Q at [384,512).
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 128;              // query rows per cluster
constexpr int kQChunkBytes = 128 * 128;  // 128 rows x 128 B
constexpr int kKvChunkBytes = 64 * 128;  // 64 tokens x 128 B
constexpr int kPeHalfBytes = 64 * 64;    // 64 tokens x 32 k_pe columns in bf16 (64-byte rows)
constexpr int kMaxStages = 5;  // page stages in the ring (at most)
constexpr int kSinQuadBytes = 32 * 32 * 4;    // peer's partial S: 32 rows x 32 tokens of one quadrant
constexpr int kSinBytes = 4 * kSinQuadBytes;
constexpr int kPBytes = kRows * 128;    // P[128 rows x 64 tokens] bf16
constexpr int kPHalfBytes = kPBytes / 2;  // one token half of P
constexpr int kStageOff = 0;
constexpr int kCtlBytes = 2048;

// Shared-memory layout.  Each CTA holds four c_kv chunks and half of k_pe (32
// columns, 64-byte swizzled rows) of every page in bf16 (f16 with an FP8
// cache), so QK^T is 18 MMAs in both CTAs.  With an FP8 cache the e4m3 codes
// land at stage + 16 KB (below) and the converter writes the f16 tiles over
// the whole stage.
template <bool kFp8>
struct Layout {
  static constexpr int kStageBytes = 4 * kKvChunkBytes + kPeHalfBytes;
  static constexpr int kStages = 4;                                  // page stages in the ring
  // Q's c_kv chunks land in the last two stages' space, then go to TMEM.
  static constexpr int kQStageOff = kStageOff + (kStages - 2) * kStageBytes;
  static constexpr int kSinOff = kStageOff + kStages * kStageBytes;  // S_in: the peer's partial scores, per quadrant
  static constexpr int kSoutOff = kSinOff + kSinBytes;               // S_out: partial scores staged for the peer
  static constexpr int kPBufs = 2;                                   // P buffers
  static constexpr int kPOff = kSoutOff + kSinBytes;
  static constexpr int kQpeOff = kPOff + kPBufs * kPBytes;           // q_pe columns (A from shared memory)
  static constexpr int kQpeBytes = kQChunkBytes / 2;
  static constexpr int kCtlOff = kQpeOff + kQpeBytes;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;    // + alignment slack
  static_assert(4 * kQChunkBytes <= 2 * kStageBytes, "Q staging");
  static_assert(kStages >= 3 && kStages <= kMaxStages, "stages");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kPOff % 1024 == 0 && kQpeOff % 1024 == 0, "swizzle atoms");
};

// FP8 cache: the CTA's 256 e4m3 c_kv columns of a page land 128B-swizzled as
// two 8 KB boxes at stage + 16 KB, the space of f16 chunks 2 and 3, and its 32
// e4m3 k_pe columns 32B-swizzled at stage + 32 KB, under the f16 k_pe tile.
// FP8 query (kQ8): QK^T runs on those codes themselves (tcgen05 kind::f8f6f4),
// so the converter writes chunks 2-3 only once QK of the page has completed and
// never touches the k_pe codes (k_pe only enters QK).  The query's c_kv columns
// sit in tensor memory four codes per column, its 32 q_pe codes per row in
// shared memory (32B swizzle).
constexpr int kQ8RawOff = 16 * 1024;
constexpr int kQ8RawPeOff = 32 * 1024;
constexpr int kQ8Box = 64 * 128;     // 64 tokens x 128 e4m3 columns
constexpr int kQ8PeBox = 64 * 32;    // 64 tokens x 32 e4m3 k_pe columns
constexpr int kQ8QpeBytes = 128 * 32;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O_c: 256 columns
constexpr uint32_t kColS = 256;  // S: two 64-column buffers
constexpr uint32_t kColQ = 384;  // Q's c_kv chunks as the A operand: 2 bf16 per column, 128 columns

constexpr int kSoftmaxWarp0 = 2;
constexpr int kConvWarp0 = 6;    // FP8 converter warps 6-9
template <bool kFp8>
__host__ __device__ constexpr int send_warp0() { return kFp8 ? 10 : 6; }  // S sender warps
template <bool kFp8>
__host__ __device__ constexpr int pv_warp() { return kFp8 ? 14 : 10; }
template <bool kFp8>
__host__ __device__ constexpr int block_threads() { return 32 * (pv_warp<kFp8>() + 1); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far above any legitimate wait
// After an abort a CTA lingers this long before the final cluster barrier, so
// that bulk copies and st.async stores it or its peer issued before giving up
// (a few KB each, microseconds in flight) have landed before either CTA exits.
constexpr uint64_t kAbortSettleNs = 200000ull;

constexpr uint32_t kIdescQK = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescQK8 = idesc_e4m3(128, 64);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);
// FP8 cache: an e4m3 pair widens to f16 in one conversion (to bf16 it takes
// four), so the FP8-cache instances run their bf16-shaped MMAs on f16 operands:
// the cache's codes, P, and (with a bf16 query) Q and q_pe converted once per
// cluster.  Every e4m3 value is exact in f16, P (at most 2^8) gains three
// mantissa bits, and a bf16 query is exact in f16 within +-65504 (beyond that
// the request is reported as an input error).  A and B always share the type.
constexpr uint32_t kIdescQKh = idesc_f16(128, 64, false, false);
constexpr uint32_t kIdescPVh = idesc_f16(128, 256, false, true);

// Bytes the peer's warp of a quadrant delivers per page: its 32 rows' P halves
// (64 B each) into pv_ready, and the references they are computed with (4 B
// each) into u_ready.
constexpr uint32_t kPvReadyTx = 32 * 64;
constexpr uint32_t kUReadyTx = 32 * 4;

struct Ctl {
  uint64_t q_full;
  uint64_t raw_full[kMaxStages];
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];     // this CTA's PV of the stage's page has completed
  uint64_t q_tmem;             // Q moved from shared to tensor memory (count 4)
  uint64_t s_full[2];          // QK^T of the page is in TMEM
  uint64_t s_free[2];          // the live softmax and sender warps have read it (count 2 x live quadrants)
  uint64_t sin_full[4];        // per quadrant: the peer's partial S landed (count 1 + 4 KB of st.async bytes)
  uint64_t sin_free[4];        // per quadrant: the peer consumed what this CTA sent (count 1, remote)
  uint64_t p_free[2];          // PV done in both CTAs: that P buffer rewritable (count 2)
  uint64_t pv_ready[2];        // local P halves written (count: live quadrants) + the peer's halves landed
  uint64_t u_ready[2];         // the peer's references for the page landed (count: live quadrants + 128 B each)
  uint64_t checked[2];         // the live local warps ran the page's reference check (count: live quadrants)
  uint64_t p_recv[4];          // per quadrant: the peer holds this CTA's P rows it had to scale (count 1, remote)
  uint64_t qk_done[kMaxStages];  // FP8 query: QK^T of the stage's page completed (its e4m3 bytes are free)
  uint64_t fin;                // the peer's row sums delivered (count 4 + 512 B)
  uint64_t drain;
  uint32_t tmem_base;
  int req;                     // the request this cluster works on
  int abort;
  int poisoned;
  float u_peer[2][kRows];      // [P buffer][row]: reference the peer computed its half with
  float l_peer[kRows];         // the peer's exp sums at the end
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

// Two e4m3 codes (low byte first) -> two f16 values, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Two floats -> the MMA operand pair: bf16 (bf16 cache) or f16 (FP8 cache).
template <bool kHalf>
__device__ __forceinline__ uint32_t pack_pair(float a, float b) {
  if constexpr (kHalf) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
template <bool kHalf>
__device__ __forceinline__ float2 unpack_pair(uint32_t w) {
  if constexpr (kHalf)
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  else
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// A P pair times a power of two f <= 1 (f16: in half precision, where an f
// below the smallest subnormal rounds to 0 like the products it would give).
template <bool kHalf>
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float f) {
  if constexpr (kHalf) {
    __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&w), __float2half2_rn(f));
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    const float2 x = unpack_pair<false>(w);
    return pack_pair<false>(x.x * f, x.y * f);
  }
}

// A bf16 pair -> an f16 pair (exact within +-65504; `big` is set for a value
// that would round to infinity).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& big) {
  const float a = __uint_as_float(w << 16), b = __uint_as_float(w & 0xFFFF0000u);
  big |= fabsf(a) >= 65520.f || fabsf(b) >= 65520.f;
  return pack_pair<true>(a, b);
}

// Request b uses the splits whose chunk starts before its L tokens, at least
// one and at most the plan's: s_b = clamp(ceil(L / chunk), 1, splits).  The two
// questions the kernel asks of s_b, without a division:
//   does split s lie past the request's end (s >= s_b)?
__device__ __forceinline__ bool split_past_end(const DecodeParams& p, int s, int L) {
  return s > 0 && (int64_t)s * p.chunk_tokens >= L;
}
//   does the request use a single split (s_b == 1)?
__device__ __forceinline__ bool single_split(const DecodeParams& p, int L) {
  return p.splits == 1 || L <= p.chunk_tokens;
}
// The same count by division.  The FP8-cache instances keep this form: with
// the division-free tests their code lands so that their hot loops miss more
// in the instruction cache (FP8 query: no-instruction stalls 1.05 -> 1.44 per
// issue, 530 -> 579 us per call on the FP8 workload; bf16 query: 648 -> 657
// us), while the bf16-cache instance gains 1 % from them.  Measured, not
// derived: the placement is the compiler's.
__device__ __forceinline__ int request_splits(const DecodeParams& p, int L) {
  return (int)max((int64_t)1, min((int64_t)p.splits, ((int64_t)L + p.chunk_tokens - 1) / p.chunk_tokens));
}

// TMEM lane quadrants holding at least one query row of the cluster's row
// group.  With fewer than 128 rows (few heads, short MTP) the softmax and
// sender warps of the other quadrants take no part in the page loop: their
// rows are never written, so their scores and P are neither exchanged nor
// computed, which cuts the pair's per-page traffic by the same factor.
// Recomputed where needed rather than kept in a register across the kernel.
__device__ __forceinline__ int live_quads(const DecodeParams& p) {
  return min(4, (min(kRows, p.rows - (int)(blockIdx.x >> 1) * kRows) + 31) >> 5);
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
  const uint64_t limit = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (test()) return true;
    if (*(volatile int*)&c->abort) return false;
    if (globaltimer_ns() - t0 > limit) {
      *(volatile int*)&c->abort = 1;
      report_error(p.err, MLA_ERR_TIMEOUT, c->req, where, blockIdx.y);
      return false;
    }
  }
}

template <bool kFp8, bool kQ8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(block_threads<kFp8>(), 1)
    split_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                       const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kv3,
                       const __grid_constant__ CUtensorMap tm_kpe, const DecodeParams p) {
  static_assert(kFp8 || !kQ8, "an FP8 query needs the FP8 cache");
  using Lay = Layout<kFp8>;
  constexpr int kStageBytes = Lay::kStageBytes;
  constexpr int kNS = Lay::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + Lay::kCtlOff);
  uint8_t* sQ = smem + Lay::kQStageOff;  // Q staging (then the ring's last two stages)
  uint8_t* sKV = smem + kStageOff;
  uint8_t* sSin = smem + Lay::kSinOff;
  uint8_t* sQpe = smem + Lay::kQpeOff;
  uint8_t* sSout = smem + Lay::kSoutOff;
  uint8_t* sP = smem + Lay::kPOff;

  constexpr int kPvWarp = pv_warp<kFp8>();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();  // 0 or 1: which column half this CTA holds
  const uint32_t peer = cta ^ 1u;
  const int g0 = cta == 0 ? 0 : 4;         // first global chunk
  const int rg = blockIdx.x >> 1;          // row group
  const int split = blockIdx.y;

  // The lengths are fetched first (each thread one, more for big batches) so
  // that their latency overlaps the barrier set-up and the TMEM allocation,
  // which do not depend on the request.
  const bool lpt = p.order_by_length != 0;
  const int nb4 = (p.batch + 3) >> 2;  // lengths padded with INT_MIN, which never outranks anything
  const int my_len = (lpt && (int)threadIdx.x < p.batch) ? p.seq_lens[threadIdx.x] : INT_MIN;
  if (threadIdx.x == 0) {
    const int nq = live_quads(p);
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&ctl->raw_full[s], 1);
      mbar_init(&ctl->full[s], kFp8 ? 4 : 1);
      mbar_init(&ctl->empty[s], 1);
      mbar_init(&ctl->qk_done[s], 1);
    }
    mbar_init(&ctl->q_tmem, 4);
    mbar_init(&ctl->s_full[0], 1);
    mbar_init(&ctl->s_full[1], 1);
    mbar_init(&ctl->s_free[0], 2 * nq);  // live softmax and sender warps
    mbar_init(&ctl->s_free[1], 2 * nq);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&ctl->sin_full[q], 1);
      mbar_init(&ctl->sin_free[q], 1);
      mbar_init(&ctl->p_recv[q], 1);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(&ctl->pv_ready[e], nq);
      mbar_init(&ctl->checked[e], nq);
      mbar_init(&ctl->u_ready[e], nq);
    }
    mbar_init(&ctl->p_free[0], 2);
    mbar_init(&ctl->p_free[1], 2);
    mbar_init(&ctl->fin, 4);
    mbar_init(&ctl->drain, 2);  // both MMA-issuing threads' last commits
    ctl->abort = 0;
    fence_mbarrier_init();
  }

  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }

  // Clusters take the requests in order of decreasing length (ties by index):
  // the hardware starts clusters in grid order, so the longest requests start
  // first and the short ones fill the last waves (longest processing time
  // first).  The lengths are ranked in shared memory (the P buffer, idle until
  // the page loop).  The host turns this off for batches above
  // kMaxOrderedBatch and for grids that start in a single wave.
  int* lens = reinterpret_cast<int*>(sP);
  if (lpt) {
    if ((int)threadIdx.x < 4 * nb4) lens[threadIdx.x] = my_len;
    for (int i = threadIdx.x + blockDim.x; i < 4 * nb4; i += blockDim.x) lens[i] = i < p.batch ? p.seq_lens[i] : INT_MIN;
  }
  __syncthreads();
  if (lpt) {
    for (int c = threadIdx.x; c < p.batch; c += blockDim.x) {
      const int lc = lens[c];
      int rank = 0;
#pragma unroll 4
      for (int k4 = 0; k4 < nb4; ++k4) {
        const int4 l4 = reinterpret_cast<const int4*>(lens)[k4];
        const int k = 4 * k4;
        rank += (l4.x > lc) | ((l4.x == lc) & (k < c));
        rank += (l4.y > lc) | ((l4.y == lc) & (k + 1 < c));
        rank += (l4.z > lc) | ((l4.z == lc) & (k + 2 < c));
        rank += (l4.w > lc) | ((l4.w == lc) & (k + 3 < c));
      }
      if (rank == (int)blockIdx.z) ctl->req = c;
    }
  } else if (threadIdx.x == 0) {
    ctl->req = blockIdx.z;
  }
  __syncthreads();
  const int b = ctl->req;

  const int L = lpt ? lens[b] : p.seq_lens[b];  // tokens of request b in this cache
  const int row0 = rg * kRows;
  // Splits of this request: those whose chunk starts before L (at least one,
  // at most the plan's).  With a single one the cluster of split 0 writes the
  // final out/lse itself; a split past the request's end only marks its
  // partial rows empty for the combine (their outputs are never read) and
  // leaves.  The combine applies the same rule.
  if (kFp8 ? split >= request_splits(p, L) : split_past_end(p, split, L)) {
    if (cta == 0 && (int)threadIdx.x < min(kRows, p.rows - row0))
      p.partials[(((int64_t)b * p.rows + row0 + threadIdx.x) * p.splits + split) * kPartRow + kKvLora] = -INFINITY;
    if (warp == 0) tmem_dealloc(ctl->tmem_base, kTmemCols);
    return;
  }
  // This request's query tokens: rows (b, i, h) with i >= qlb are padding of a
  // per-request q_len call, computed fully masked (out 0, lse -inf).
  const int qlb = p.q_lens ? p.q_lens[b] : p.q_len;
  // A sequence shard holds positions [kv0, kv0 + L) of a request of length
  // Ltot (possibly none of them); otherwise the cache holds [0, L) and Ltot = L.
  const bool shard = p.kv_start != nullptr;
  const int kv0 = shard ? p.kv_start[b] : 0;
  const int Ltot = shard ? p.total_lens[b] : L;
  const bool q_ok = qlb >= 1 && qlb <= p.q_len;
  const bool range_ok = kv0 >= 0 && L >= 0 && (int64_t)kv0 + L <= Ltot;
  const bool len_ok = q_ok && range_ok && Ltot >= qlb && L <= p.max_seq_len;
  const int lo = split * p.chunk_tokens;
  const int hi = len_ok ? min(lo + p.chunk_tokens, L) : lo;
  const int first_page = lo / kPage;
  const int n_pages = hi > lo ? (hi + kPage - 1) / kPage - first_page : 0;
  const float kv_scale = (kFp8 && p.kv_scale) ? *p.kv_scale : 1.0f;
  const float q_scale = (kQ8 && p.q_scale) ? *p.q_scale : 1.0f;  // folded into the softmax scale
  const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride + first_page;

  // Thread 0 is the TMA producer: it starts Q's loads (into this CTA's own
  // shared memory, on a barrier it initialised itself) and the first
  // block-table lookup before the cluster-wide sync.
  int page_first = 0;
  if (threadIdx.x == 0) {
    ctl->poisoned = len_ok ? 0 : 1;
    if (!len_ok && split == 0 && rg == 0 && cta == 0)  // index -2: q_len, -3: shard range, -1: length
      report_error(p.err, MLA_ERR_DEVICE_INPUT, b, !q_ok ? -2 : (!range_ok ? -3 : -1),
                   !q_ok ? qlb : (!range_ok ? kv0 : L));
    if (n_pages > 0) {
      page_first = bt_row[0];
      fence_proxy_async_smem();  // the barrier initialisations are visible to the copy engine
      prefetch_tmap(&tm_qn);
      prefetch_tmap(&tm_qp);
      const int qrow = b * p.rows + row0;
      if (kQ8) {  // two 128-code boxes of the CTA's c_kv columns, and its 32 q_pe codes
        mbar_arrive_expect_tx(&ctl->q_full, 2 * kQChunkBytes + kQ8QpeBytes);
        for (int k = 0; k < 2; ++k)
          tma_load_2d(sQ + k * kQChunkBytes, &tm_qn, &ctl->q_full, 256 * (int)cta + 128 * k, qrow);
      } else {
        mbar_arrive_expect_tx(&ctl->q_full, 4 * kQChunkBytes + kQChunkBytes / 2);
        for (int k = 0; k < 4; ++k) tma_load_2d(sQ + k * kQChunkBytes, &tm_qn, &ctl->q_full, (g0 + k) * 64, qrow);
      }
      tma_load_2d(sQpe, &tm_qp, &ctl->q_full, 32 * (int)cta, qrow);
      prefetch_tmap(&tm_kv);
      if (!kFp8) prefetch_tmap(&tm_kv3);
      prefetch_tmap(&tm_kpe);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_pages > 0) {  // Q is on its way (see above)
      int issued = 0;
      int next_page = page_first;
      for (int j = 0; j < n_pages; ++j) {
        const int s = j % kNS;
        const int page = next_page;
        if (j + 1 < n_pages) next_page = bt_row[j + 1];  // lookups ahead of the waits
        // The last two stages hold Q until the softmax warps have moved it into TMEM.
        if (j == kNS - 2 && !wait_bar(ctl, &ctl->q_tmem, 0, p, 17)) break;
        if (!wait_bar(ctl, &ctl->empty[s], ((j / kNS) & 1) ^ 1, p, 1)) break;
        uint64_t* land = kFp8 ? &ctl->raw_full[s] : &ctl->full[s];
        uint8_t* stage = sKV + s * kStageBytes;
        if (page < 0 || page >= p.num_pages) {
          if (cta == 0) report_error(p.err, MLA_ERR_DEVICE_INPUT, b, first_page + j, page);
          mbar_arrive(land);  // nothing to load; consumers mask the whole page
        } else if (kFp8) {  // e4m3: two 128B-swizzled boxes of 128 c_kv codes, one 32B-swizzled k_pe box
          mbar_arrive_expect_tx(land, 2 * kQ8Box + kQ8PeBox);
          for (int k = 0; k < 2; ++k)
            tma_load_2d(stage + kQ8RawOff + k * kQ8Box, &tm_kv, land, 256 * (int)cta + 128 * k, page * kPage);
          tma_load_2d(stage + kQ8RawPeOff, &tm_kpe, land, 8 * 64 + 32 * (int)cta, page * kPage);
        } else {
          // The CTA's four c_kv chunks in one 3-D box (columns x rows x chunks),
          // which lands as [chunk][row][128 B], and its 32 k_pe columns in a 2-D
          // box with 64-byte swizzled rows.
          mbar_arrive_expect_tx(land, 4 * kKvChunkBytes + kPeHalfBytes);
          tma_load_3d(stage, &tm_kv3, land, 0, page * kPage, g0);
          tma_load_2d(stage + 4 * kKvChunkBytes, &tm_kpe, land, 8 * 64 + 32 * (int)cta, page * kPage);
        }
        issued = j + 1;
      }
      // Never leave with copies in flight.
      for (int j = max(0, issued - kNS); j < issued; ++j) {
        uint64_t* land = kFp8 ? &ctl->raw_full[j % kNS] : &ctl->full[j % kNS];
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(land), (j / kNS) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK^T issuer
    // QK(j) as soon as page j has landed and its S buffer is free.  PV has a
    // thread of its own (below), so a PV that becomes ready never waits behind
    // the issue of a QK; the stage ring, S, S_in and P barriers bound how far QK
    // runs ahead.
    if constexpr (kQ8) {
     if (lane == 0 && n_pages > 0) {
      // FP8 query: QK(j) on the page's e4m3 codes as soon as they land (the
      // converter's f16 V is only needed by PV): 8 K-steps of 32 codes over the
      // two c_kv boxes, A from tensor memory, and one over the 32 k_pe codes, A
      // (q_pe) from shared memory.  qk_done tells the converter that the codes
      // under V chunks 2 and 3 may be overwritten.
      const uint32_t kv_addr = smem_u32(sKV);
      const uint64_t qpe_desc = sdesc_sw32(smem_u32(sQpe), 16, 256);
      bool ok = wait_bar(ctl, &ctl->q_tmem, 0, p, 2);
      for (int j = 0; ok && j < n_pages; ++j) {
        const int st = j % kNS;
        if (!wait_bar(ctl, &ctl->raw_full[st], (j / kNS) & 1, p, 3) ||
            !wait_bar(ctl, &ctl->s_free[j & 1], ((j >> 1) & 1) ^ 1, p, 4))
          break;
        tc_fence_after();
        const uint32_t stage = kv_addr + st * kStageBytes;
        const uint32_t d = tmem + kColS + (j & 1) * 64;
        for (int k = 0; k < 2; ++k) {
          const uint64_t k_desc = sdesc_sw128(stage + kQ8RawOff + k * kQ8Box, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 32 codes per K-step: 32 bytes of the swizzled row, 8 TMEM columns
            mma_f8_ts(d, tmem + kColQ + k * 32 + kk * 8, k_desc + (uint64_t)((kk * 32) >> 4), kIdescQK8,
                      (k | kk) ? 1u : 0u);
        }
        mma_f8_ss(d, qpe_desc, sdesc_sw32(stage + kQ8RawPeOff, 16, 256), kIdescQK8, 1u);
        mma_commit(&ctl->s_full[j & 1]);
        mma_commit(&ctl->qk_done[st]);
      }
      mma_commit(&ctl->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
     }
    } else if (lane == 0 && n_pages > 0) {
      const uint32_t kv_addr = smem_u32(sKV);
      const uint64_t qpe_desc = sdesc_sw64(smem_u32(sQpe), 16, 512);
      bool ok = wait_bar(ctl, &ctl->q_tmem, 0, p, 2);
      for (int j = 0; ok && j < n_pages; ++j) {
        if (!wait_bar(ctl, &ctl->full[j % kNS], (j / kNS) & 1, p, 3) ||
            !wait_bar(ctl, &ctl->s_free[j & 1], ((j >> 1) & 1) ^ 1, p, 4))
          break;
        tc_fence_after();
        const uint64_t k_desc = sdesc_sw128(kv_addr + (j % kNS) * kStageBytes, 16, 1024);
        const uint32_t d = tmem + kColS + (j & 1) * 64;
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A = Q chunk k from TMEM: 16 k per MMA = 8 columns
            mma_16b_ts(d, tmem + kColQ + k * 32 + kk * 8, k_desc + (uint64_t)((k * kKvChunkBytes + kk * 32) >> 4),
                        kFp8 ? kIdescQKh : kIdescQK, (k | kk) ? 1u : 0u);
        }
        {  // this CTA's 32 k_pe columns: two K-steps along 64-byte swizzled rows
          const uint64_t kpe_desc = sdesc_sw64(kv_addr + (j % kNS) * kStageBytes + 4 * kKvChunkBytes, 16, 512);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_16b_ss(d, qpe_desc + (uint64_t)((kk * 32) >> 4), kpe_desc + (uint64_t)((kk * 32) >> 4),
                       kFp8 ? kIdescQKh : kIdescQK, 1u);
        }
        mma_commit(&ctl->s_full[j & 1]);
      }
      mma_commit(&ctl->drain);  // every MMA of this thread has completed before TMEM is freed
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // PV(j) in two halves of 32 tokens: this CTA's own half as soon as the local
    // warps have checked page j's references (which they do after writing their
    // P rows, scaling O or P where the references moved), the peer's half once
    // its P rows have landed.  The own half runs while the peer's are in flight.
    if (lane == 0 && n_pages > 0) {
      const uint32_t kv_addr = smem_u32(sKV);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = true;
      for (int j = 0; ok && j < n_pages; ++j) {
        if (!wait_bar(ctl, &ctl->checked[j & 1], (j >> 1) & 1, p, 7)) break;
        // With an FP8 query QK(j) did not wait for the converter: V must be in.
        if (kQ8 && !wait_bar(ctl, &ctl->full[j % kNS], (j / kNS) & 1, p, 24)) break;
        tc_fence_after();
        const int pb = j % Lay::kPBufs;
        const uint64_t v_desc = sdesc_sw128(kv_addr + (j % kNS) * kStageBytes, kKvChunkBytes, 1024);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int h = i == 0 ? (int)cta : (int)peer;  // token half
          if (i == 1) {
            if (!wait_bar(ctl, &ctl->pv_ready[j & 1], (j >> 1) & 1, p, 5)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {  // A = P tokens 16kk..16kk+15: two 8-token chunks of half h
            const int kk = 2 * h + t;
            mma_16b_ss(tmem + kColO,
                        sdesc_noswz(p_addr + pb * kPBytes + h * kPHalfBytes + ((2 * kk) & 3) * 128, 128, 512),
                        v_desc + (uint64_t)((kk * 2048) >> 4), kFp8 ? kIdescPVh : kIdescPV,
                        (j > 0 || i > 0 || t > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(&ctl->empty[j % kNS]);           // stage free; O current through page j
        mma_commit_multicast(&ctl->p_free[pb], 3);  // P buffer reusable, in both CTAs
      }
      mma_commit(&ctl->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  } else if (kFp8 && warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
    // ------------------------------------------------------------ e4m3 -> f16 converter
    // The CTA's 256 c_kv codes of a page land as two 128B-swizzled boxes of 128
    // codes at stage + 16 KB.  Thread ct takes token t = ct%64 of box h = ct/64
    // (eight 16-byte units) into f16 chunks 2h and 2h+1 (128B swizzle): a warp's
    // loads and stores cover eight distinct units per eight lanes, free of bank
    // conflicts.  Box 1's codes lie under chunks 2-3, so every thread holds its
    // codes before any is rewritten.
    //   bf16 query: QK^T needs f16 K as well, so the 32 k_pe codes (32B-swizzled
    //     at stage + 32 KB, under the f16 k_pe tile) are widened too, half a
    //     token row per thread.  V rows past L are zeroed by the softmax warps.
    //   FP8 query: QK^T reads the codes themselves, so box 1's warps wait for
    //     QK of the page before writing chunks 2-3, and the converter writes
    //     zeros for tokens at or past L and for a page that was never loaded.
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    const int t = ct & 63, h = ct >> 6;
    const int tp = ct >> 1, hp = ct & 1;           // bf16 query: k_pe token and 16-code half
    int page_next = n_pages > 0 ? bt_row[0] : 0;
    for (int j = 0; j < n_pages; ++j) {
      const int st = j % kNS;
      bool zero = false;
      if constexpr (kQ8) {
        const int page = page_next;
        if (j + 1 < n_pages) page_next = bt_row[j + 1];
        const bool page_ok = page >= 0 && page < p.num_pages;
        zero = t >= (page_ok ? min(L - (lo + j * kPage), kPage) : 0);
      }
      if (conv_sync_or(!wait_bar(ctl, &ctl->raw_full[st], (j / kNS) & 1, p, 9))) break;
      uint8_t* stage = sKV + st * kStageBytes;
      uint4 raw[8], rpe;
      const uint8_t* src = stage + kQ8RawOff + h * kQ8Box + t * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) raw[u] = *reinterpret_cast<const uint4*>(src + ((u ^ (t & 7)) << 4));
      if constexpr (!kQ8)  // 32B swizzle: the 16-byte unit flips with bit 2 of the row
        rpe = *reinterpret_cast<const uint4*>(stage + kQ8RawPeOff + tp * 32 + ((hp ^ ((tp >> 2) & 1)) << 4));
      bool ok = true;
      if constexpr (kQ8) {
        conv_sync();  // every thread holds its codes before box 1's space is rewritten
        ok = h == 0 || __all_sync(0xffffffffu, wait_bar(ctl, &ctl->qk_done[st], (j / kNS) & 1, p, 25));
      } else {
        conv_sync();  // every thread holds its codes (c_kv and k_pe) before any is rewritten
      }
      // Logical 16-code piece u of the row: f16 chunk 2h + u/4, 16-byte units
      // 2(u%4) and 2(u%4)+1 of token row t (128B swizzle).
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint8_t* dst = stage + (2 * h + (u >> 2)) * kKvChunkBytes + t * 128;
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          o[2 * q] = zero ? 0u : e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu));
          o[2 * q + 1] = zero ? 0u : e4m3x2_to_f16x2((uint16_t)(w[q] >> 16));
        }
        const int c0 = 2 * (u & 3);
        *reinterpret_cast<uint4*>(dst + ((c0 ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + (((c0 + 1) ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      if constexpr (!kQ8) {  // k_pe: 16 codes -> units 2hp, 2hp+1 of the 64B-swizzled f16 row tp
        uint8_t* dst = stage + 4 * kKvChunkBytes + tp * 64;
        const uint32_t w[4] = {rpe.x, rpe.y, rpe.z, rpe.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          o[2 * q] = e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu));
          o[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(w[q] >> 16));
        }
        *reinterpret_cast<uint4*>(dst + (((2 * hp) ^ ((tp >> 1) & 3)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + (((2 * hp + 1) ^ ((tp >> 1) & 3)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      if constexpr (kQ8) {
        if (conv_sync_or(!ok)) break;
      }
      fence_proxy_async_smem();
      conv_sync();
      if (lane == 0) mbar_arrive(&ctl->full[st]);
    }
  } else if (warp >= send_warp0<kFp8>() && warp < send_warp0<kFp8>() + 4) {
    // ------------------------------------------------------------ S sender
    // The peer's token half of S(j), for the rows of TMEM lane quadrant w%4, goes
    // from TMEM through S_out to the peer's S_in as one 4 KB bulk copy, as soon as
    // QK(j) is done and the peer has consumed the previous page's partial (which
    // also means the previous copy has read S_out).  Off the softmax warps' chain,
    // the peer's partial is in place before the softmax warps come to it.
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t col_oth = kColS + 32 * peer;
    uint8_t* sout_quad = sSout + quad * kSinQuadBytes;
    uint8_t* sout_row = sout_quad + lane * 128;
    const uint32_t sin_quad_peer = mapa_shared(smem_u32(sSin + quad * kSinQuadBytes), peer);
    const uint32_t sin_full_peer = mapa_shared(smem_u32(&ctl->sin_full[quad]), peer);
    const int n_send = quad < live_quads(p) ? n_pages : 0;
    for (int j = 0; j < n_send; ++j) {
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->s_full[sb], (j >> 1) & 1, p, 20))) break;
      tc_fence_after();
      uint32_t oth[2][16];
      tmem_ld16(tmem + lane_base + col_oth + sb * 64, oth[0]);
      tmem_ld16(tmem + lane_base + col_oth + sb * 64 + 16, oth[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free[sb]);
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->sin_free[quad], (j & 1) ^ 1, p, 13))) break;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(sout_row + ((u ^ (lane & 7)) << 4)) =
            make_uint4(oth[u >> 2][(u & 3) * 4], oth[u >> 2][(u & 3) * 4 + 1], oth[u >> 2][(u & 3) * 4 + 2],
                       oth[u >> 2][(u & 3) * 4 + 3]);
      fence_proxy_async_smem();  // staged rows visible to the copy engine
      __syncwarp();
      if (lane == 0) bulk_copy_to_peer(sin_quad_peer, sout_quad, kSinQuadBytes, sin_full_peer);
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ------------------------------------------------------------ softmax / exchange warpgroup
    // Each CTA owns one half of every page's 64 tokens (CTA c: tokens 32c..32c+31)
    // for all 128 rows; warp w handles the rows of TMEM lane quadrant w%4.  Per
    // page a warp hands the peer the partial scores of the peer's token half,
    // adds the peer's partial for its own half, and computes P for its half, which
    // it writes into both CTAs' P buffers.  Order within page j: add the peer's
    // partial of S(j); settle and send the reference; P(j) out; check page j;
    // own half of S(j+1) from TMEM.  P(j) and the check come first so that PV(j),
    // and with it the release of page j's stage for the next load, is not held
    // up by the next page.
    //
    // Reference maxima.  P of one row must share one reference across both
    // halves, yet neither CTA sees the other's scores.  Each CTA computes with
    // its own reference r_ref (a whole number in the exp2 domain, so that any two
    // differ by a power of two), raised lazily to ceil(max) when a score exceeds
    // it by more than 2^8.  With every P half goes the reference it used; once
    // both halves of page k are in, each CTA takes the larger of the two and of
    // the previous agreed value, scales O if the agreed value moved, and scales
    // any P half computed against a lower reference (a raise, or a reference the
    // CTA had not yet learnt from its peer) before PV(k).  Outside of raises,
    // which occur on a split's first pages and when a row's max jumps, that check
    // touches nothing.
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // row within the group (TMEM lane)
    const bool row_ok = row0 + r < p.rows;   // the row exists (it is written)
    const int qi = (row0 + r) / p.num_heads;
    const bool row_live = row_ok && qi < qlb;  // not padding of a per-request q_len
    // Tokens of this cache the row may see: its causal limit in this cache's
    // positions, and never past the cache's own L (a shard's range can end
    // before the row's limit).
    const int vis = min(Ltot - qlb + 1 + qi - kv0, L);
    const float sc2 = p.softmax_scale * kv_scale * q_scale * kLog2e;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t col_own = kColS + 32 * cta;    // S columns of this CTA's token half (within a buffer)
    uint8_t* sin_row = sSin + quad * kSinQuadBytes + lane * 128;  // 32 fp32 of the peer's partial
    const uint32_t sin_free_peer = mapa_shared(smem_u32(&ctl->sin_free[quad]), peer);
    const uint32_t p_peer = mapa_shared(smem_u32(sP), peer);
    float r_ref = -INFINITY;   // reference this CTA computes P with
    float a_ref = -INFINITY;   // reference both CTAs agreed on, through the last checked page
    float l_sum = 0.f;         // exp sum over this CTA's token halves, relative to r_ref
    int own_fixes = 0;         // pages on which this warp scaled its own P rows (p_recv phases)
    bool poisoned = !len_ok;
    bool q_bad = false;        // this row's query does not fit the FP8-cache path's f16 operands
    bool ok = true;

    // 16-byte chunk u (tokens 8u..8u+7) of this thread's row of P.  P is K-major
    // without swizzle, laid out [token half][8-row group][8-token chunk][row][16 B],
    // so a warp's 32 rows of one token half are 2 KB of contiguous bytes.
    auto p_chunk = [&](int pb, int u) -> uint8_t* {
      return sP + pb * kPBytes + (u >> 2) * kPHalfBytes + (r >> 3) * 512 + (u & 3) * 128 + (r & 7) * 16;
    };
    const int p_mine_off = (int)cta * kPHalfBytes + quad * 2048;  // this warp's rows of this CTA's half

    // This CTA's token half of S(jj) from TMEM into `own` (the sender warps
    // take the peer's half).
    auto take_s = [&](int jj, float (&own)[32]) -> bool {
      const int sb = jj & 1;
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->s_full[sb], (jj >> 1) & 1, p, 6))) return false;
      tc_fence_after();
      uint32_t mine[2][16];
      tmem_ld16(tmem + lane_base + col_own + sb * 64, mine[0]);
      tmem_ld16(tmem + lane_base + col_own + sb * 64 + 16, mine[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free[sb]);
#pragma unroll
      for (int k = 0; k < 32; ++k) own[k] = __uint_as_float(mine[k >> 4][k & 15]);
      return true;
    };

    // Page k's reference check, run once the peer's references for page k are in
    // and before PV(k) may be issued (the MMA waits for `checked`).  Only when a
    // P half must be scaled does it also wait for the peer's P halves.
    auto check = [&](int k, float u_own) -> bool {
      const int e = k & 1;
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->u_ready[e], (k >> 1) & 1, p, 11))) return false;
      const float u_oth = ctl->u_peer[e][r];
      const float an = fmaxf(a_ref, fmaxf(u_own, u_oth));
      const bool resc = k > 0 && an > a_ref;  // PV(0) overwrites O
      const bool fix_own = u_own < an, fix_oth = u_oth < an;
      const bool any_own = __any_sync(0xffffffffu, fix_own), any_oth = __any_sync(0xffffffffu, fix_oth);
      if (__any_sync(0xffffffffu, resc) || any_own || any_oth) {
        if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->pv_ready[e], (k >> 1) & 1, p, 19))) return false;
        if (__any_sync(0xffffffffu, resc)) {
          // O holds exactly pages < k once PV(k-1) has completed.
          if (!__all_sync(0xffffffffu,
                          wait_bar(ctl, &ctl->empty[(k - 1) % kNS], ((k - 1) / kNS) & 1, p, 12)))
            return false;
          tc_fence_after();
          const float f = resc ? ex2(a_ref - an) : 1.f;
#pragma unroll 1
          for (int g = 0; g < 16; ++g) {
            uint32_t v[16];
            const uint32_t ta = tmem + lane_base + kColO + g * 16;
            tmem_ld16(ta, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
            tmem_st16(ta, v);
          }
          tmem_st_wait();
          tc_fence_before();
        }
        // P halves computed against a lower reference; the factors are powers of
        // two.  The peer's half first: its rows have landed (pv_ready), so the
        // peer learns that its copy is done with its source and may scale that
        // half in place.  This CTA's own half was sent to the peer just before
        // this check; it is scaled in place only once the peer signals the same,
        // so that the copy never reads half-scaled rows.  Both CTAs take the same
        // decisions (an, the references and a_ref are equal on both sides).
        auto scale_half = [&](int h, bool fix, float u) {
          if (!fix) return;
          const float f = ex2(u - an);
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            uint4* c = reinterpret_cast<uint4*>(p_chunk(k % Lay::kPBufs, 4 * h + uu));
            uint4 w = *c;
            uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              wv[i] = scale_pair<kFp8>(wv[i], f);
            }
            *c = w;
          }
        };
        if (any_oth) {
          scale_half((int)peer, fix_oth, u_oth);
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&ctl->p_recv[quad]), peer));
        }
        if (any_own) {
          if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->p_recv[quad], own_fixes & 1, p, 23))) return false;
          ++own_fixes;
          scale_half((int)cta, fix_own, u_own);
        }
        fence_proxy_async_smem();
      }
      if (an > r_ref) {
        l_sum *= ex2(r_ref - an);
        r_ref = an;
      }
      a_ref = an;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->checked[e]);
      return true;
    };

    // Q_c rows into tensor memory: thread = row = TMEM lane; the 128B-swizzled
    // staging rows are un-swizzled into 2-bf16 columns, 32 columns per chunk.
    if (n_pages > 0) {
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->q_full, 0, p, 18))) {
        ok = false;
      } else {
        // bf16: four 64-column chunks (2 per TMEM column); FP8: two 128-code
        // chunks (4 per column).  Either way a chunk row is 128 bytes.  With an
        // FP8 cache and a bf16 query the values become f16 on the way (the
        // MMAs' operand type there), and so do the row's q_pe values in place.
        bool big = false;
        for (int k = 0; k < (kQ8 ? 2 : 4); ++k) {
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
          if constexpr (kFp8 && !kQ8) {
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i >> 4][i & 15] = bf16x2_to_f16x2(w[i >> 4][i & 15], big);
          }
          tmem_st16(tmem + lane_base + kColQ + k * 32, w[0]);
          tmem_st16(tmem + lane_base + kColQ + k * 32 + 16, w[1]);
        }
        if constexpr (kFp8 && !kQ8) {  // the row's 32 q_pe values: 64 bytes (swizzle stays inside the row)
          uint4* qp = reinterpret_cast<uint4*>(sQpe + r * 64);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v = qp[u];
            v.x = bf16x2_to_f16x2(v.x, big);
            v.y = bf16x2_to_f16x2(v.y, big);
            v.z = bf16x2_to_f16x2(v.z, big);
            v.w = bf16x2_to_f16x2(v.w, big);
            qp[u] = v;
          }
          fence_proxy_async_smem();  // the f16 q_pe is what the QK issuer's MMAs read
          if (big && row_ok) {  // index -4: a query value outside the f16 range of this path
            q_bad = true;
            report_error(p.err, MLA_ERR_DEVICE_INPUT, b, -4, row0 + r);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->q_tmem);
    }

    // Block-table entries are loaded one page ahead: a global load consumed in
    // the same iteration would stall every page for a full memory latency.
    int page_next = n_pages > 0 ? bt_row[0] : 0;
    float sv_next[32];
    const bool live = quad < live_quads(p);  // (the group's other warps go straight to the epilogue)
    if (ok && live && n_pages > 0 && !take_s(0, sv_next)) ok = false;
    for (int j = 0; ok && live && j < n_pages; ++j) {
      const int e = j & 1;   // pv_ready / checked / peer references of this page
      const int tok0 = lo + j * kPage;  // lo is page aligned
      const int page = page_next;
      if (j + 1 < n_pages) page_next = bt_row[j + 1];
      const bool page_ok = page >= 0 && page < p.num_pages;
      poisoned |= !page_ok;
      float sv[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) sv[k] = sv_next[k];

      // The peer's partial of this CTA's token half.  Pages that every row of the
      // warp sees in full (all but a split's last page, normally) take a fast
      // path: add and max on raw scores (the scale is positive, so max commutes
      // with it), then p = 2^(s*scale - ref) in one FMA + ex2.  Other pages mask
      // and scale first; masked columns, possibly NaN garbage, become -inf and
      // then exactly 0.
      if (lane == 0) mbar_arrive_expect_tx(&ctl->sin_full[quad], kSinQuadBytes);
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->sin_full[quad], j & 1, p, 14))) {
        ok = false;
        break;
      }
      const int tok_c = tok0 + 32 * (int)cta;
      const int n_vis = (page_ok && row_live) ? min(max(vis - tok_c, 0), 32) : 0;
      const bool fast = __all_sync(0xffffffffu, n_vis == 32);
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      {
        const float4* src = reinterpret_cast<const float4*>(sin_row);
        if (fast) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 v = src[u ^ (lane & 7)];
            sv[4 * u] += v.x;
            sv[4 * u + 1] += v.y;
            sv[4 * u + 2] += v.z;
            sv[4 * u + 3] += v.w;
#pragma unroll
            for (int k = 0; k < 4; ++k) mq[k] = fmaxf(mq[k], sv[4 * u + k]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 v = src[u ^ (lane & 7)];
            const float a[4] = {sv[4 * u] + v.x, sv[4 * u + 1] + v.y, sv[4 * u + 2] + v.z, sv[4 * u + 3] + v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x = (4 * u + k < n_vis) ? a[k] * sc2 : -INFINITY;
              sv[4 * u + k] = x;
              mq[k] = fmaxf(mq[k], x);
            }
          }
        }
      }
      float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      if (fast) mx *= sc2;
      __syncwarp();  // every lane's S_in values are in registers
      if (lane == 0) mbar_arrive_cluster_relaxed(sin_free_peer);

      // This page's reference is settled and goes to the peer first, ahead of
      // the larger transfers, so that the peer's check of this page need not
      // wait for them.
      if (mx > r_ref + kRescaleThreshold) {  // false while every column is masked
        const float u = ceilf(mx);
        l_sum *= ex2(r_ref - u);
        r_ref = u;
      }
      const float u_cur = r_ref;
      st_async_u32(mapa_shared(smem_u32(&ctl->u_peer[e][r]), peer), __float_as_uint(u_cur),
                   mapa_shared(smem_u32(&ctl->u_ready[e]), peer));
      if (lane == 0) mbar_arrive_expect_tx(&ctl->u_ready[e], kUReadyTx);


      // V rows of tokens at or past L (or of a page that was never loaded) may
      // hold anything, NaN included; zero this CTA's 256 V columns of them (64
      // tokens x four 128-byte chunk rows, shared among the live warps' threads).
      const int n_valid = page_ok ? min(L - tok0, kPage) : 0;
      if (!kQ8 && n_valid < kPage) {  // (with an FP8 query the converter writes those rows as zeros)
        uint8_t* stage = sKV + (j % kNS) * kStageBytes;
        const int step = 32 * live_quads(p);
        for (int i = r; i < kPage * 4; i += step) {
          const int t = i >> 2;
          if (t >= n_valid) {
            uint4* rowp = reinterpret_cast<uint4*>(stage + (i & 3) * kKvChunkBytes + t * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) rowp[u] = make_uint4(0, 0, 0, 0);
          }
        }
      }

      uint4 pk[4];
      float part[4] = {0.f, 0.f, 0.f, 0.f};
      if (fast) {
        const float nm = -r_ref;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float p0 = ex2(fmaf(sv[u * 8 + 2 * h], sc2, nm));
            const float p1 = ex2(fmaf(sv[u * 8 + 2 * h + 1], sc2, nm));
            part[h] += p0 + p1;
            w[h] = pack_pair<kFp8>(p0, p1);
          }
          pk[u] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float x0 = sv[u * 8 + 2 * h], x1 = sv[u * 8 + 2 * h + 1];
            const float p0 = (x0 == -INFINITY) ? 0.f : ex2(x0 - r_ref);
            const float p1 = (x1 == -INFINITY) ? 0.f : ex2(x1 - r_ref);
            part[h] += p0 + p1;
            w[h] = pack_pair<kFp8>(p0, p1);
          }
          pk[u] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      l_sum += (part[0] + part[1]) + (part[2] + part[3]);

      // Both CTAs' PV of the page that last used this P buffer must be done.
      const int pb = j % Lay::kPBufs;
      if (!__all_sync(0xffffffffu, wait_bar(ctl, &ctl->p_free[pb], ((j / Lay::kPBufs) & 1) ^ 1, p, 15))) {
        ok = false;
        break;
      }
      // The warp's P rows go to the peer as one 2 KB bulk copy (the copy engine
      // carries them; the warp does not stall on the pair's link).
#pragma unroll
      for (int u = 0; u < 4; ++u) *reinterpret_cast<uint4*>(p_chunk(pb, 4 * (int)cta + u)) = pk[u];
      fence_proxy_async_smem();  // P rows (and any zeroed V rows) visible to the MMA and the copy engine
      __syncwarp();
      const uint32_t pv_bar_peer = mapa_shared(smem_u32(&ctl->pv_ready[e]), peer);
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->pv_ready[e], kPvReadyTx);
        const int off = pb * kPBytes + p_mine_off;
        bulk_copy_to_peer(p_peer + (uint32_t)off, sP + off, 2048, pv_bar_peer);
      }
      // Then this page's reference check, after which PV(j) may go (the own
      // half at once, the peer's half when its P is in), and the own half of the
      // next page's scores.
      if (!check(j, u_cur)) {
        ok = false;
        break;
      }
      if (j + 1 < n_pages && !take_s(j + 1, sv_next)) {
        ok = false;
        break;
      }
    }
    ok = !wg_sync_or(!ok);  // the epilogue decides as one group

    // ------------------------------------------------------------ epilogue
    // Row sums of both token halves: every row's partial goes to the peer.
    // (NaN marks a row whose query this CTA found out of range: the peer writes
    // it as NaN too.)
    st_async_u32(mapa_shared(smem_u32(&ctl->l_peer[r]), peer), __float_as_uint(q_bad ? NAN : l_sum),
                 mapa_shared(smem_u32(&ctl->fin), peer));
    if (lane == 0) mbar_arrive_expect_tx(&ctl->fin, 32 * 4);
    if (poisoned) atomicOr(&ctl->poisoned, 1);
    bool fail = !wait_bar(ctl, &ctl->fin, 0, p, 16);
    fail |= !ok || (n_pages > 0 && !wait_bar(ctl, &ctl->empty[(n_pages - 1) % kNS], ((n_pages - 1) / kNS) & 1, p, 8));
    fail = wg_sync_or(fail);
    tc_fence_after();
    __syncwarp();
    const bool have_o = !fail && n_pages > 0;
    const bool bad = ctl->poisoned != 0 || fail || (kFp8 && !kQ8 && (q_bad || ctl->l_peer[r] != ctl->l_peer[r]));
    const float l_tot = l_sum + ctl->l_peer[r];
    const bool has = l_tot > 0.f;
    const float il = has ? kv_scale / l_tot : 0.f;
    const int64_t grow0 = (int64_t)b * p.rows + row0;
    const bool one_split = kFp8 ? request_splits(p, L) == 1 : single_split(p, L);
    if (cta == 0 && row_ok) {
      const float lv = bad ? NAN : (has ? (r_ref + lg2(l_tot)) * kLn2 : -INFINITY);
      if (one_split) {
        if (p.lse) p.lse[(grow0 + r) * p.lse_stride] = lv;
        // +inf (never a real LSE) in split 0's slot: the combine leaves the row alone
        if (p.splits > 1) p.partials[(grow0 + r) * p.splits * kPartRow + kKvLora] = INFINITY;
      } else {
        p.partials[((grow0 + r) * p.splits + split) * kPartRow + kKvLora] = lv;
      }
    }
    const int rows_here = min(kRows, p.rows - row0);
    // O_c rows are TMEM lanes: each warp stages 32 rows x 32 columns at a time
    // through shared memory (S_out and P, idle once the last PV has completed) so
    // that the global stores run along the columns.  The next chunk's TMEM load is
    // in flight while a chunk is written out.
    constexpr int kTileStride = 36;  // floats per staged row: 16-byte stores free of bank conflicts
    float* tile = reinterpret_cast<float*>(sSout) + (warp - kSoftmaxWarp0) * (32 * kTileStride);
    uint32_t v[2][16];
    if (have_o) {
      tmem_ld16(tmem + lane_base + kColO, v[0]);
      tmem_ld16(tmem + lane_base + kColO + 16, v[1]);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < 256; c0 += 32) {
      float4 f[8];
      if (have_o) {
        tmem_ld_wait();
        const float sc = il > 0.f ? il : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          f[u] = make_float4(__uint_as_float(v[u >> 2][(u & 3) * 4]) * sc, __uint_as_float(v[u >> 2][(u & 3) * 4 + 1]) * sc,
                             __uint_as_float(v[u >> 2][(u & 3) * 4 + 2]) * sc,
                             __uint_as_float(v[u >> 2][(u & 3) * 4 + 3]) * sc);
        if (c0 + 32 < 256) {
          tmem_ld16(tmem + lane_base + kColO + c0 + 32, v[0]);
          tmem_ld16(tmem + lane_base + kColO + c0 + 48, v[1]);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (bad) {
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = make_float4(NAN, NAN, NAN, NAN);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) *reinterpret_cast<float4*>(tile + lane * kTileStride + 4 * u) = f[u];
      __syncwarp();
      // Lane l writes column c0+l of the warp's 32 rows: one coalesced 128-byte
      // row segment per store, addresses stepping by a constant row stride.  All
      // 32 staged values are read first: with the loads interleaved, each would
      // wait out the previous store (the compiler cannot tell the two apart).
      float col[32];
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) col[rr] = tile[rr * kTileStride + lane];
      __syncwarp();  // the tile may be rewritten once every lane holds its column
      const int dim = (int)cta * 256 + c0 + lane;
      const int nr = min(32, rows_here - quad * 32);  // rows of this warp that exist
      if (!one_split) {
        float* dst = p.partials + ((grow0 + quad * 32) * p.splits + split) * kPartRow + dim;
        const int64_t step = (int64_t)p.splits * kPartRow;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          if (rr < nr) dst[rr * step] = col[rr];
      } else if (p.out_fp32 && p.out_stride == kKvLora) {
        float* dst = reinterpret_cast<float*>(p.out) + (grow0 + quad * 32) * kKvLora + dim;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          if (rr < nr) dst[rr * kKvLora] = col[rr];
      } else if (p.out_fp32) {  // 513-wide partial rows of a sequence shard
        float* dst = reinterpret_cast<float*>(p.out) + (grow0 + quad * 32) * p.out_stride + dim;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          if (rr < nr) dst[rr * p.out_stride] = col[rr];
      } else if (p.out_fp8) {  // (bf16 and e4m3 outputs always have 512-wide rows)
        const float osc = p.out_scale ? *p.out_scale : 1.f;
        uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) + (grow0 + quad * 32) * kKvLora + dim;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          if (rr < nr) dst[rr * kKvLora] = to_e4m3(col[rr], osc);
      } else {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + (grow0 + quad * 32) * kKvLora + dim;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          if (rr < nr) dst[rr * kKvLora] = __float2bfloat16_rn(col[rr]);
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0 && *(volatile int*)&ctl->abort) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kAbortSettleNs) {
    }
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

// 2-D tensor map: `rows` rows of `cols` elements, `stride_elems` apart, box box_cols x box_rows.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_elems,
               CUtensorMapDataType dt, uint32_t elem_bytes, uint32_t box_rows, CUtensorMapSwizzle swz,
               uint32_t box_cols = 64) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride_elems * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map over a bf16 cache: {64 columns, rows, 9 chunks of 64 columns},
// box {64, 64 rows, 4 chunks}, 128-byte swizzle.  The chunk dimension steps back
// through each row (stride 128 B), so one box lands as four 8 KB chunk tiles.
bool encode_kv_chunks(CUtensorMap* m, const void* base, uint64_t rows) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, rows, kRow / 64};
  cuuint64_t strides[2] = {(cuuint64_t)kRow * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kPage, 4};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kFp8, bool kQ8>
cudaError_t launch_kernel(const dim3& grid, const CUtensorMap& tm_qn, const CUtensorMap& tm_qp,
                          const CUtensorMap& tm_kv, const CUtensorMap& tm_kv3, const CUtensorMap& tm_kpe,
                          const DecodeParams& p, cudaStream_t stream) {
  auto kern = split_kv_tc_kernel<kFp8, kQ8>;
  constexpr int kSmem = Layout<kFp8>::kSmemBytes;
  // The shared-memory opt-in is a property of the kernel in the device's
  // context: set once per device (a bit per device; a lost race only repeats
  // the same idempotent call).
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  kern<<<grid, block_threads<kFp8>(), kSmem, stream>>>(tm_qn, tm_qp, tm_kv, tm_kv3, tm_kpe, p);
  return cudaGetLastError();
}

// FP8 query: tensor maps over e4m3 codes, boxes shaped for QK^T on the codes
// (128B swizzle for c_kv, 32B swizzle for the 32 rope codes of each CTA).
cudaError_t launch_split_kv_q8(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap tm_qn, tm_qp, tm_kv, tm_kpe;
  const uint64_t q_rows = (uint64_t)p.batch * p.rows;
  const uint64_t kv_rows = (uint64_t)p.num_pages * kPage;
  if (!encode_2d(&tm_qn, p.q_nope, kKvLora, q_rows, p.q_nope_stride, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B, 128) ||
      !encode_2d(&tm_qp, p.q_pe, kRope, q_rows, p.q_pe_stride, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128,
                 CU_TENSOR_MAP_SWIZZLE_32B, 32) ||
      !encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                 128) ||
      !encode_2d(&tm_kpe, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64, CU_TENSOR_MAP_SWIZZLE_32B,
                 32))
    return cudaErrorInvalidValue;
  const dim3 grid(2 * p.row_groups, p.splits, p.batch);
  return launch_kernel<true, true>(grid, tm_qn, tm_qp, tm_kv, tm_kv, tm_kpe, p, stream);
}

}  // namespace

cudaError_t launch_split_kv(const DecodeParams& p, cudaStream_t stream) {
  if (p.q_fp8) return p.kv_fp8 ? launch_split_kv_q8(p, stream) : cudaErrorInvalidValue;
  CUtensorMap tm_qn, tm_qp, tm_kv, tm_kv3, tm_kpe;
  const uint64_t q_rows = (uint64_t)p.batch * p.rows;
  const uint64_t kv_rows = (uint64_t)p.num_pages * kPage;
  if (!encode_2d(&tm_qn, p.q_nope, kKvLora, q_rows, p.q_nope_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_qp, p.q_pe, kRope, q_rows, p.q_pe_stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128,
                 CU_TENSOR_MAP_SWIZZLE_64B, 32))
    return cudaErrorInvalidValue;
  const bool ok = p.kv_fp8 ? encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64,
                                       CU_TENSOR_MAP_SWIZZLE_128B, 128)
                           : encode_2d(&tm_kv, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  // bf16 cache viewed as [chunk 0..8][row][64 columns]: row stride 1152 B, chunk stride 128 B.
  if (!p.kv_fp8 && !encode_kv_chunks(&tm_kv3, p.kv, kv_rows)) return cudaErrorInvalidValue;
  // 32 k_pe columns per box: bf16 with 64-byte swizzled rows, or 32 e4m3 bytes
  // with 32-byte swizzled rows.
  if (!(p.kv_fp8 ? encode_2d(&tm_kpe, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64,
                             CU_TENSOR_MAP_SWIZZLE_32B, 32)
                 : encode_2d(&tm_kpe, p.kv, kRow, kv_rows, kRow, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64,
                             CU_TENSOR_MAP_SWIZZLE_64B, 32)))
    return cudaErrorInvalidValue;
  if (p.kv_fp8) tm_kv3 = tm_kv;  // unused on the FP8 path
  const dim3 grid(2 * p.row_groups, p.splits, p.batch);
  if (p.kv_fp8) return launch_kernel<true, false>(grid, tm_qn, tm_qp, tm_kv, tm_kv3, tm_kpe, p, stream);
  return launch_kernel<false, false>(grid, tm_qn, tm_qp, tm_kv, tm_kv3, tm_kpe, p, stream);
}

}  // namespace mla
