// Sparse MLA decode, Eq. (2) of "DeepSeek V3.2-Exp support" (llama.cpp issue
// 16331, section "1. Architecture"): attention of each query row's 128 heads
// over only the k selected latents c_s (576 = 512 latent + 64 rope elements;
// the value is the first 512).
//
// Work unit = a cluster of two CTAs per (row, split); 128 selected tokens per
// tile.  The pair divides the work by operand instead of by output columns, so
// every selected latent crosses into the pair's shared memory once for S and
// once for P V, and S is computed once:
//
//  CTA 0, the score CTA (TMEM: two S tiles [128 heads x 128 tokens] f32 at
//  columns 0-127 and 128-255, so S(i+1) is computed while the softmax reads
//  S(i); elements 0-511 of Q at 256-511, lane = head, two bf16 per column; Q's
//  rope elements 512-575 stay in shared memory as the A operand of the last
//  K-chunk):
//   warps 0-7  gather the nine [128 tokens x 64] K-chunks of each tile (16-byte
//              cp.async, manual 128-byte swizzle, a skipped selection is
//              zero-filled; completion by cp.async.mbarrier.arrive, so no
//              gathering thread waits) into a 9-slot ring, one slot per chunk;
//   warps 8-11 softmax, one thread per head: Q -> TMEM once (by TMA into
//              ring slots 0-7 before the gathers start, then each thread
//              moves its head's row; the gathers' cp.async path is left to
//              the gathers); per tile read S twice (its maximum, then P),
//              mask skipped selections, keep a lazily moving reference (it
//              moves only when a score exceeds it by more than 2^8), write P
//              as bf16 into a K-major 128B-swizzled message buffer with the
//              tile's O correction factors and running sums (one local
//              message buffer, rewritten once the copy has read it);
//   warp 12    tcgen05 issuer of S = Q K^T (kind::f16, A = Q from TMEM,
//              M = 128 heads, N = 128 tokens, K = 576);
//   warp 13    sends each tile's message once the four softmax warps have
//              written it, and frees the local buffer when the copy has read
//              it, so the softmax warps never wait on the copy engine.
//  CTA 1, the value CTA (TMEM: O [128 heads x 512] f32, all 512 columns):
//   warps 0-7  gather the eight [128 tokens x 64] value chunks of each tile
//              (the latent lines the score CTA read a tile earlier: L2 hits);
//   warps 8-11 rescale O when a message says the reference moved, and write
//              the normalised output at the end;
//   warp 12    tcgen05 issuer of O += P V (A = P from the message, K-major;
//              V MN-major from the ring, N = 256 per four chunks), whose
//              completion frees the message buffer in both CTAs (multicast
//              commit) and the ring slots.
// With more than one split the pair writes unnormalised partial O plus its
// (max, sum) and a combine kernel merges them.
//
// Measured on GB300: a lone thread issuing bf16 MMAs (M = 128, K = 16) in a
// tight loop is held 64 cycles per MMA for N <= 128 and 128 at N = 256 (so
// P V issues N = 256), and every instruction between its MMAs adds to that,
// hence descriptors formed as base + constant offset.  A tile then costs the
// score CTA ~6 k cycles at the ~1.6 GHz the SMs run at during this kernel in
// the decode step: its 144 KB of 16-byte gathers (~24.5 B/cycle per SM), with
// the S / softmax / P V chain close behind.  With one S tile the next tile's
// MMAs waited for the softmax to read S; with two they do not.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kSoftWarp = kGatherWarps;     // warps 8-11: softmax (CTA 0) / O warps (CTA 1)
constexpr int kMmaWarp = kGatherWarps + 4;  // warp 12: MMA issuer; owns the TMEM allocation
constexpr int kSendWarp = kMmaWarp + 1;     // warp 13: message sender (CTA 0)
constexpr int kThreads = 32 * (kSendWarp + 1);
constexpr int kTile = 128;
constexpr int kChunksS = 9;  // 576 / 64: K-chunks per tile (score CTA)
constexpr int kChunksV = 8;  // 512 / 64: value chunks per tile (value CTA)
constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kHalf = 256;   // columns of one partial-O block of the combine kernel
constexpr uint32_t kChunkBytes = kTile * 128;  // 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// TMEM columns.
constexpr uint32_t kSCol = 0;    // score CTA: S tiles (2 x 128 columns)
constexpr uint32_t kQCol = 256;  // score CTA: Q elements 0-511 (256 columns)
constexpr uint32_t kTmemCols = 512;

// Message score CTA -> value CTA for one tile: P [128 heads x 128 tokens] bf16
// as two K-major 128B-swizzled chunks (tokens 0-63, 64-127), the factor O
// must be multiplied by before this tile's P V, the running sum after it, and
// one "reference moved" flag per softmax warp.
constexpr uint32_t kMsgCorr = 2 * kChunkBytes;
constexpr uint32_t kMsgL = kMsgCorr + 4 * kHeads;
constexpr uint32_t kMsgFlags = kMsgL + 4 * kHeads;
constexpr uint32_t kMsgBytes = kMsgFlags + 16;
constexpr uint32_t kMsgStride = 34 * 1024;  // keeps the P chunks 1024-byte aligned
static_assert(kMsgBytes <= kMsgStride && kMsgBytes % 16 == 0, "message layout");

// Shared memory: a header of barriers at the same offset in both CTAs (the
// multicast commit names a barrier by its offset), then each CTA's payload.
struct Header {
  uint64_t full[kChunksS], empty[kChunksS];  // ring slots (one per chunk of a tile)
  uint64_t s_full[2], s_free[2];             // score CTA: S tile b written / read
  uint64_t q_ready;                          // score CTA: Q in TMEM
  uint64_t p_full[2], p_free[2];             // message buffer b: arrived / consumed by P V
  uint64_t need_fix, o_fixed, drain;         // value CTA: O rescale hand-off, final drain
  uint64_t q_full;                           // score CTA: a round of Q chunks landed
  uint64_t msg_ready[2], msg_free[2];        // score CTA: message part written / read by its copy
  uint32_t tmem_base;
  int abort;
  int t_fix;  // tile whose P V waits for an O rescale, or -1 = no more tiles
};
constexpr uint32_t kHeaderBytes = 1024;
static_assert(sizeof(Header) <= kHeaderBytes, "header");
constexpr uint32_t kScoreRing = 0;
constexpr uint32_t kScoreMsg = kChunksS * kChunkBytes;
constexpr uint32_t kScoreRope = kScoreMsg + kMsgStride;  // Q elements 512-575, [128 x 64]
constexpr uint32_t kValueMsg = 0;
constexpr uint32_t kValueRing = 2 * kMsgStride;
constexpr uint32_t kScorePayload = kScoreRope + kChunkBytes;
static_assert(kScoreRope % 1024 == 0, "128B-swizzled operands are 1024-byte aligned");
constexpr uint32_t kValuePayload = kValueRing + kChunksV * kChunkBytes;
constexpr uint32_t kPayloadBytes = kScorePayload > kValuePayload ? kScorePayload : kValuePayload;
constexpr size_t kSmemBytes = 1024 + kHeaderBytes + kPayloadBytes;
static_assert(kSmemBytes <= 227 * 1024, "sparse MLA shared memory exceeds 227 KB");

struct MParams {
  const uint16_t* q;  // [R, 128, 576] bf16
  const uint8_t* kv;  // latent cache base: row r (page*64 + slot) at kv + r * 1152
  const int32_t* bt;
  int64_t bt_stride;
  int num_pages;
  int next_n;
  const int32_t* row_bt;  // null, or [R]: the block-table row of each query row
  int bt_num_rows;        // with row_bt: the rows of the block table
  const int32_t* idx;
  int k;
  float scale_log2;
  int nsplit;
  int tokens_per_split;
  uint16_t* out;
  float* lse;
  float* ws;  // partials when nsplit > 1
  uint32_t* err;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}


// 2^x by the hardware approximation (a few ulp; P is rounded to bf16 anyway).
// 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Partial block of (row, value half vh, split) for the combine kernel:
// 128 x 256 O, then 128 maxima, then 128 sums.
__device__ __forceinline__ float* partial_block(const MParams& p, int row, int vh, int split) {
  return p.ws + ((static_cast<int64_t>(row) * 2 + vh) * p.nsplit + split) *
                    (kHeads * kHalf + 2 * kHeads);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const MParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Header& s = *reinterpret_cast<Header*>(base);
  uint8_t* pay = base + kHeaderBytes;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = score CTA, 1 = value CTA
  // The setup reads no global memory, so it runs before the wait for the
  // previous kernel: barriers, TMEM, the pair's first cluster barrier.
  if (tid == 0) {
    s.abort = 0;
    s.t_fix = 0;
    for (int i = 0; i < kChunksS; ++i) {
      mbar_init(&s.full[i], 32 * kGatherWarps);  // one cp.async completion per gather thread
      mbar_init(&s.empty[i], 1);                 // the MMA issuer's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.s_full[b], 1);
      mbar_init(&s.s_free[b], 4);  // the 4 softmax warps have read S tile b
    }
    mbar_init(&s.q_ready, 4);  // the 4 softmax warps have stored their Q rows
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.p_full[b], 1);  // the score CTA's remote arrive (+ the copy's bytes)
      mbar_init(&s.p_free[b], 1);  // the value CTA's multicast commit
    }
    mbar_init(&s.need_fix, 1);
    mbar_init(&s.o_fixed, 4);
    mbar_init(&s.drain, 1);
    mbar_init(&s.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.msg_ready[b], 4);  // the 4 softmax warps have written part b of the message
      mbar_init(&s.msg_free[b], 1);   // the sender's copy has read part b
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  // both CTAs' barriers are initialised before any remote arrival or copy
  cluster_sync_all();
  tc_fence_after();
  pdl_launch_dependents_and_wait();
  const int row = blockIdx.x >> 1;
  const int split = blockIdx.y;
  // the block-table row of this query row (an out-of-range one reads nothing)
  int req = p.row_bt ? p.row_bt[row] : row / p.next_n;
  if (p.row_bt && (req < 0 || req >= p.bt_num_rows)) {
    if (tid == 0 && rank == 0) raise_error(p.err, kErrBadPage);
    req = -1;
  }
  const int s0 = split * p.tokens_per_split;
  const int s1 = min(p.k, s0 + p.tokens_per_split);
  const int ntile = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(row) * p.k;

  volatile int* abort = &s.abort;
  const uint32_t tmem = s.tmem_base;

  if (warp < kGatherWarps) {
    // -------------------------------------------------------------- gather --
    const int nch = rank == 0 ? kChunksS : kChunksV;
    uint8_t* ring = pay + (rank == 0 ? kScoreRing : kValueRing);
    const int gt = tid;  // 0 .. 32*kGatherWarps-1
    // Thread gt copies, of every 16 KB chunk, the 16-byte pieces gt + 256 q
    // (q = 0..3): chunk row (gt >> 3) + 32 q, piece gt & 7.  Its 4 latent rows
    // (page*64 + slot, -1 = skipped) of tile i+1 are computed while tile i is
    // issued: idx is read two tiles ahead, the block table one tile ahead.
    constexpr int kRowStep = (32 * kGatherWarps) / 8;  // 32 rows between a thread's pieces
    const int prow = gt >> 3, pch = gt & 7;
    auto load_toks = [&](int i, int (&t)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = s0 + i * kTile + prow + kRowStep * u;
        t[u] = (i < ntile && pos < s1) ? idx_row[pos] : -1;
      }
    };
    auto load_pages = [&](const int (&t)[4], int (&pg)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t pg_i = t[u] / 64;
        pg[u] = (t[u] >= 0 && pg_i < p.bt_stride)
                    ? (req >= 0 ? p.bt[static_cast<int64_t>(req) * p.bt_stride + pg_i] : -1) : -1;
      }
    };
    auto make_rows = [&](const int (&t)[4], const int (&pg)[4], int (&r)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        r[u] = -1;
        if (t[u] >= 0) {
          if (pg[u] >= 0 && pg[u] < p.num_pages) r[u] = pg[u] * 64 + t[u] % 64;
          else if (pch == 0 && rank == 0) raise_error(p.err, kErrBadIndex);
        }
      }
    };
    int tk_next[4], rows_cur[4];
    {
      int t0[4], pg0[4];
      load_toks(0, t0);
      load_pages(t0, pg0);
      make_rows(t0, pg0, rows_cur);
      load_toks(1, tk_next);
    }
    bool bad = false;
    // the score CTA's ring holds Q's staging until Q is in TMEM
    if (rank == 0 && ntile > 0 && !mbar_wait_warp(&s.q_ready, 0, p.err, abort)) bad = true;
    for (int i = 0; i < ntile && !bad; ++i) {
      // loads for the next tiles go out first; their results are used after
      // this tile's copies have been issued
      int pg_next[4] = {-1, -1, -1, -1}, tk_after[4] = {-1, -1, -1, -1};
      if (i + 1 < ntile) {
        load_pages(tk_next, pg_next);
        load_toks(i + 2, tk_after);
      }
      for (int c = 0; c < nch; ++c) {
        // slot c held chunk c of tile i-1 until its MMAs completed
        if (i > 0 && !mbar_wait_warp(&s.empty[c], (i - 1) & 1, p.err, abort)) { bad = true; break; }
        uint8_t* dst = ring + c * kChunkBytes;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint8_t* d = dst + sw128_offset(prow + kRowStep * u, pch);
          if (rows_cur[u] >= 0)
            cp_async_16(d, p.kv + static_cast<int64_t>(rows_cur[u]) * (kDqk * 2) + c * 128 + pch * 16);
          else
            cp_async_16_zero(d, p.kv);
        }
        cp_async_mbar_arrive_noinc(&s.full[c]);
      }
      int rows_next[4] = {-1, -1, -1, -1};
      if (i + 1 < ntile) make_rows(tk_next, pg_next, rows_next);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        rows_cur[u] = rows_next[u];
        tk_next[u] = tk_after[u];
      }
    }
    cp_async_wait<0>();  // no copy of this thread is left in flight at exit
  } else if (warp == kMmaWarp) {
    if (rank == 0) {
      // ------------------------------------------------------ S MMA issuer --
      // One thread; S(i) goes to S tile i & 1 once the softmax has read S(i-2).
      constexpr uint32_t kIdescS = make_idesc(1, 1, 128, kTile, false, false);
      // The issuing thread shares its SM sub-partition with a softmax and two
      // gather warps, so its loop is kept short: descriptors are the base
      // ones plus constant offsets (the start-address field holds address
      // >> 4 in 14 bits, and no operand ends above 256 KB, so adding to it
      // never carries into the next field).
      const uint64_t ring_desc = sw128_desc(smem_u32(pay + kScoreRing), 16, 1024);
      const uint64_t rope_desc = sw128_desc(smem_u32(pay + kScoreRope), 16, 1024);
      if (lane == 0 && ntile > 0 && mbar_wait(&s.q_ready, 0, p.err, abort)) {
        tc_fence_after();
        for (int i = 0; i < ntile && !*abort; ++i) {
          const int sb = i & 1;
          if (i >= 2 && !mbar_wait(&s.s_free[sb], ((i - 2) >> 1) & 1, p.err, abort)) break;
          tc_fence_after();
          const uint32_t d = tmem + kSCol + kTile * sb;
          bool bad = false;
#pragma unroll
          for (int c = 0; c < kChunksS; ++c) {
            if (!mbar_wait(&s.full[c], i & 1, p.err, abort)) { bad = true; break; }
            fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core
            tc_fence_after();
            // chunk c of the ring; a K step of 16 elements is 32 bytes
            const uint64_t bd = ring_desc + static_cast<uint64_t>(c * (kChunkBytes >> 4));
            if (c < kChunksV) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ts(d, tmem + kQCol + 32 * c + 8 * kk, bd + 2 * kk, kIdescS, (c | kk) != 0);
            } else {
              // the rope elements: A = Q's [128 x 64] rope chunk in shared memory
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) mma_f16(d, rope_desc + 2 * kk, bd + 2 * kk, kIdescS, 1u);
            }
            mma_commit(&s.empty[c]);
          }
          if (bad) break;
          mma_commit(&s.s_full[sb]);
        }
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------ PV MMA issuer --
      // O[:, 256 j4 .. +256] += P V_j4 per four value chunks j4 (N = 256);
      // each group's ring slots are freed as soon as its MMAs complete, so the
      // next tile's gathers start while this tile's second group runs.
      constexpr uint32_t kIdescPV = make_idesc(1, 1, 128, 256, false, true);
      const uint8_t* msg0 = pay + kValueMsg;
      // as for S: base descriptors plus constant offsets (no carry out of the
      // 14-bit start-address field below 256 KB)
      const uint64_t v_desc = sw128_desc(smem_u32(pay + kValueRing), kChunkBytes, 1024);
      if (lane == 0) {
        int nfix = 0;
        for (int t = 0; t < ntile && !*abort; ++t) {
          const int b = t & 1;
          const uint8_t* msg = msg0 + b * kMsgStride;
          if (!mbar_wait_cluster(&s.p_full[b], (t >> 1) & 1, p.err, abort)) break;
          const uint32_t* fl = reinterpret_cast<const uint32_t*>(msg + kMsgFlags);
          if ((fl[0] | fl[1] | fl[2] | fl[3]) != 0) {
            // the reference moved: O (through P V of tile t-1) is rescaled first
            *reinterpret_cast<volatile int*>(&s.t_fix) = t;
            mbar_arrive(&s.need_fix);
            if (!mbar_wait(&s.o_fixed, nfix & 1, p.err, abort)) break;
            ++nfix;
          }
          bool bad = false;
          const uint64_t p_desc = sw128_desc(smem_u32(msg), 16, 1024);
#pragma unroll
          for (int j4 = 0; j4 < kChunksV / 4; ++j4) {
            for (int c = 4 * j4; c < 4 * j4 + 4; ++c)
              if (!mbar_wait(&s.full[c], t & 1, p.err, abort)) { bad = true; break; }
            if (bad) break;
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t vd = v_desc + static_cast<uint64_t>(4 * j4 * (kChunkBytes >> 4));
            // K step kk: tokens 16 kk .. +16, i.e. P chunk kk / 4 at byte 32 (kk % 4)
            // and V rows 16 kk (2 KB further per step)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_f16(tmem + 256 * j4,
                      p_desc + static_cast<uint64_t>(((kk >> 2) * kChunkBytes + 32 * (kk & 3)) >> 4),
                      vd + static_cast<uint64_t>((2048 * kk) >> 4), kIdescPV,
                      (t > 0 || kk > 0) ? 1u : 0u);
            for (int c = 4 * j4; c < 4 * j4 + 4; ++c) mma_commit(&s.empty[c]);
          }
          if (bad) break;
          // message buffer b is free again in both CTAs once these MMAs complete
          mma_commit_mc(&s.p_free[b], 0x3);
        }
        *reinterpret_cast<volatile int*>(&s.t_fix) = -1;
        mbar_arrive(&s.need_fix);
        // every MMA of this thread (and its arrivals in the score CTA) completes
        // before the pair leaves
        mma_commit(&s.drain);
        mbar_wait(&s.drain, 0, p.err, abort);
      }
      __syncwarp();
    }
  } else if (warp == kSendWarp) {
    if (rank == 0 && lane == 0) {
      // ---------------------------------------------------- message sender --
      // Each message goes in two copies: part 0 (P of tokens 0-63) as soon as
      // it is written, part 1 (P of tokens 64-127, the factors and sums) at
      // the end of the tile; each part of the local buffer is freed when its
      // copy has read it.
      const uint32_t peer_msg0 = mapa_shared(smem_u32(pay + kValueMsg), 1);
      const uint8_t* msg = pay + kScoreMsg;
      int sent = 0;
      for (int i = 0; i < ntile; ++i) {
        const int b = i & 1;
        if (!mbar_wait(&s.msg_ready[0], i & 1, p.err, abort)) break;
        // the value CTA's buffer b is free once P V of tile i-2 has completed
        if (i >= 2 && !mbar_wait_cluster(&s.p_free[b], ((i - 2) >> 1) & 1, p.err, abort)) break;
        const uint32_t pbar = mapa_shared(smem_u32(&s.p_full[b]), 1);
        const uint32_t dst = peer_msg0 + b * kMsgStride;
        mbar_arrive_expect_tx_remote(pbar, kMsgBytes);
        bulk_copy_s2s(dst, msg, kChunkBytes, pbar);
        bulk_commit_group();
        ++sent;
        bulk_wait_group_read<0>();
        mbar_arrive(&s.msg_free[0]);
        if (!mbar_wait(&s.msg_ready[1], i & 1, p.err, abort)) break;
        bulk_copy_s2s(dst + kChunkBytes, msg + kChunkBytes, kMsgBytes - kChunkBytes, pbar);
        bulk_commit_group();
        bulk_wait_group_read<0>();
        mbar_arrive(&s.msg_free[1]);
      }
      bulk_wait_group<0>();
      // the value CTA's last commits arrive here too: they land before the pair exits
      for (int t = max(0, sent - 2); t < sent; ++t)
        if (!mbar_wait_cluster(&s.p_free[t & 1], (t >> 1) & 1, p.err, abort)) break;
    }
    __syncwarp();
  } else if (rank == 0) {
    // ----------------------------------------------------------- softmax --
    const int quad = warp & 3;       // warps 8-11: TMEM lane quadrants 0-3
    const int h = quad * 32 + lane;  // head == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const bool leader = warp == kSoftWarp && lane == 0;
    uint8_t* msg0 = pay + kScoreMsg;
    float m_run = -INFINITY, l_run = 0.f;
    bool bad = false;
    if (ntile > 0) {
      // Q elements 0-511 of the row -> TMEM columns [kQCol, kQCol + 256),
      // lane h = head h, column j holding elements 2j (low half) and 2j + 1:
      // one round of eight TMA boxes ([128 heads x 64] K-chunks, 128B-swizzled)
      // into ring slots 0-7, from which each thread copies its head's row into
      // TMEM; the gathers, whose first copies wait on two dependent index
      // loads anyway, start filling the ring once Q is in TMEM (q_ready).  The
      // round also brings the rope chunk (elements 512-575) to its own shared
      // memory.
      uint8_t* stage = pay + kScoreRing;  // 8 x 16 KB, 1024-aligned
      if (leader) tma_prefetch_desc(&tm_q);
      int q_rounds = 0;  // TMA rounds issued onto q_full
#pragma unroll 1
      for (int rd = 0; rd < 1; ++rd) {
        const int c0 = 0, nc = kChunksV;
        ++q_rounds;
        if (leader) {
          mbar_arrive_expect_tx(&s.q_full, (rd == 0 ? nc + 1 : nc) * kChunkBytes);
          for (int j = 0; j < nc; ++j)
            tma_load_2d(stage + j * kChunkBytes, &tm_q, &s.q_full, 64 * (c0 + j), row * kHeads);
          if (rd == 0)
            tma_load_2d(pay + kScoreRope, &tm_q, &s.q_full, 64 * kChunksV, row * kHeads);
        }
        __syncwarp();
        const bool ok = mbar_wait_warp(&s.q_full, rd & 1, p.err, abort);
        if (ok) {
          for (int j = 0; j < nc; ++j) {
            uint32_t r[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 w = *reinterpret_cast<const uint4*>(stage + j * kChunkBytes + sw128_offset(h, u));
              r[4 * u] = w.x;
              r[4 * u + 1] = w.y;
              r[4 * u + 2] = w.z;
              r[4 * u + 3] = w.w;
            }
            tmem_st32_sync(lane_base + kQCol + 32 * (c0 + j), r);
          }
          fence_proxy_async_smem();  // these reads come before the next round's TMA writes
        }
        // every thread has its rows before the ring slots are refilled
        if (named_bar_or(1, 128, !ok)) { bad = true; break; }
      }
      // a round whose wait ran out may still be landing: it lands before the
      // CTA can exit (at once on the normal path)
      if (leader) mbar_drain(&s.q_full, (q_rounds - 1) & 1, p.err);
      tc_fence_before();
      __syncwarp();
      if (!bad && lane == 0) mbar_arrive(&s.q_ready);
    }
    // validity of a tile's 128 selections: lane j of every warp reads entries
    // j, 32+j, 64+j, 96+j; four ballots give the tile's mask.  A selection is
    // valid if it is not -1 and its page is inside the cache: exactly the
    // selections the gather warps copy (the others are zero-filled there and
    // must get P = 0 here).  The indices are read two tiles ahead and their
    // block-table entries one tile ahead, and compared only when the tile
    // comes, so no load latency sits at the top of a tile.
    auto load_sel = [&](int i, int (&v)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = s0 + i * kTile + 32 * u + lane;
        v[u] = (i < ntile && pos < s1) ? idx_row[pos] : -1;
      }
    };
    auto load_pg = [&](const int (&v)[4], int (&pg)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pg[u] = -1;
        const int64_t pg_i = v[u] / 64;
        if (v[u] >= 0 && req >= 0 && pg_i < p.bt_stride)
          pg[u] = p.bt[static_cast<int64_t>(req) * p.bt_stride + pg_i];
      }
    };
    int sel_cur[4], pg_cur[4], sel_next[4];
    load_sel(0, sel_cur);
    load_sel(1, sel_next);
    load_pg(sel_cur, pg_cur);
    bool msg_ok = true;  // the waits for the local message buffer
    for (int i = 0; i < ntile && !bad; ++i) {
      unsigned m[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m[u] = __ballot_sync(0xffffffffu, sel_cur[u] >= 0 && pg_cur[u] >= 0 && pg_cur[u] < p.num_pages);
      int sel_after[4], pg_next[4];
      load_sel(i + 2, sel_after);
      load_pg(sel_next, pg_next);
      const bool all_valid = (m[0] & m[1] & m[2] & m[3]) == 0xffffffffu;  // warp-uniform
      const int b = i & 1;  // the value CTA's message buffer for this tile
      uint8_t* msg = msg0;
      const bool ok = mbar_wait_warp(&s.s_full[b], (i >> 1) & 1, p.err, abort);
      if (ok) tc_fence_after();
      if (named_bar_or(1, 128, !ok || !msg_ok)) { bad = true; break; }
      // Two passes over the tile's scores, 64 columns at a time.  First the
      // tile's maximum (of the raw scores: the scale is positive, so scaling
      // and rounding keep the order), then P = 2^(scale s - m_t) against the
      // running reference m_t, which moves to the tile's maximum only when
      // that exceeds it by more than the threshold (skipped selections give
      // P = 0).  Knowing m_t before any P is written lets each half of P go
      // to the value CTA as soon as it is written.
      float hm_raw = -INFINITY;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[64];
        tmem_ld64_sync(lane_base + kSCol + kTile * b + 64 * half, v);
        float h4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (all_valid) {
#pragma unroll
          for (int j = 0; j < 64; ++j) h4[j & 3] = fmaxf(h4[j & 3], v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int t = 64 * half + j;
            const bool okj = ((m[t >> 5] >> (t & 31)) & 1u) != 0;
            h4[j & 3] = fmaxf(h4[j & 3], okj ? v[j] : -INFINITY);
          }
        }
        hm_raw = fmaxf(hm_raw, fmaxf(fmaxf(h4[0], h4[1]), fmaxf(h4[2], h4[3])));
      }
      const float hm = hm_raw * p.scale_log2;  // -inf if nothing of the tile is valid
      float m_t = m_run, l_t = 0.f;
      if (hm > m_t + kRescaleThreshold || (m_t == -INFINITY && hm > -INFINITY)) m_t = hm;
      // m_t is -inf only while every score seen is -inf: those give P = 0
      const float nref = m_t == -INFINITY ? 0.f : -m_t;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[64];
        tmem_ld64_sync(lane_base + kSCol + kTile * b + 64 * half, v);
        if (half == 1) {
          // the S tile has been read: S(i+2) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.s_free[b]);
        }
        uint32_t pk[32];
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
        if (all_valid) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float e0 = ex2_approx(fmaf(v[2 * j], p.scale_log2, nref));
            const float e1 = ex2_approx(fmaf(v[2 * j + 1], p.scale_log2, nref));
            pk[j] = pack_bf16(e0, e1);
            l4[j & 3] += e0 + e1;  // the exact weights (P itself is rounded to bf16)
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int t = 64 * half + 2 * j;
            const bool ok0 = ((m[t >> 5] >> (t & 31)) & 1u) != 0;
            const bool ok1 = ((m[(t + 1) >> 5] >> ((t + 1) & 31)) & 1u) != 0;
            const float e0 = ok0 ? ex2_approx(fmaf(v[2 * j], p.scale_log2, nref)) : 0.f;
            const float e1 = ok1 ? ex2_approx(fmaf(v[2 * j + 1], p.scale_log2, nref)) : 0.f;
            pk[j] = pack_bf16(e0, e1);
            l4[j & 3] += e0 + e1;
          }
        }
        l_t += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        // part `half` of the local buffer is rewritten only after the copy of
        // tile i-1 has read it (a wait that runs out stops the softmax at the
        // next tile)
        if (i > 0 && !mbar_wait_warp(&s.msg_free[half], (i - 1) & 1, p.err, abort)) msg_ok = false;
        // row h of chunk `half`: tokens 8q .. 8q+7 of the half in 16-byte piece q
        uint8_t* chunk = msg + half * kChunkBytes;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(chunk + sw128_offset(h, q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        if (half == 0) {
          fence_proxy_async_smem();  // generic writes -> the bulk copy (async proxy)
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.msg_ready[0]);
        }
      }
      // O and l hold earlier tiles against m_run: they are brought to m_t
      const bool moved = m_t != m_run && m_run > -INFINITY;
      const float corr = moved ? ex2_approx(m_run - m_t) : 1.f;
      l_run = l_run * corr + l_t;
      m_run = m_t;
      reinterpret_cast<float*>(msg + kMsgCorr)[h] = corr;
      reinterpret_cast<float*>(msg + kMsgL)[h] = l_run;
      const bool wmoved = __any_sync(0xffffffffu, moved);
      if (lane == 0) reinterpret_cast<uint32_t*>(msg + kMsgFlags)[quad] = wmoved ? 1u : 0u;
      fence_proxy_async_smem();  // generic writes -> the bulk copy (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.msg_ready[1]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        sel_cur[u] = sel_next[u];
        pg_cur[u] = pg_next[u];
        sel_next[u] = sel_after[u];
      }
    }
    if (!msg_ok) bad = true;
    if (!bad) {
      if (p.nsplit == 1) {
        if (p.lse)
          p.lse[static_cast<int64_t>(row) * kHeads + h] =
              l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      } else {
        for (int vh = 0; vh < 2; ++vh) {
          float* blk = partial_block(p, row, vh, split);
          blk[kHeads * kHalf + h] = m_run;
          blk[kHeads * kHalf + kHeads + h] = l_run;
        }
      }
    }
  } else {
    // ------------------------------------------------- O rescale / epilogue --
    const int quad = warp & 3;
    const int h = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint8_t* msg0 = pay + kValueMsg;
    bool bad = false;
    for (int k = 0;; ++k) {
      if (!mbar_wait_warp(&s.need_fix, k & 1, p.err, abort)) { bad = true; break; }
      const int tf = *reinterpret_cast<volatile int*>(&s.t_fix);
      if (tf < 0) break;
      if (tf >= 1) {
        // O must hold P V of tile tf-1 complete before it is rescaled
        const int tp = tf - 1;
        if (!mbar_wait_warp(&s.p_free[tp & 1], (tp >> 1) & 1, p.err, abort)) { bad = true; break; }
        tc_fence_after();
        const float corr =
            reinterpret_cast<const float*>(msg0 + (tf & 1) * kMsgStride + kMsgCorr)[h];
#pragma unroll 1
        for (int cc = 0; cc < 512 / 32; ++cc) {
          float o[32];
          tmem_ld32_sync(lane_base + 32 * cc, o);
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(o[j] * corr);
          tmem_st32_sync(lane_base + 32 * cc, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.o_fixed);
    }
    if (!bad && ntile > 0) {
      const int tl = ntile - 1;
      if (mbar_wait_warp(&s.p_free[tl & 1], (tl >> 1) & 1, p.err, abort)) {
        tc_fence_after();
        const float lr = reinterpret_cast<const float*>(msg0 + (tl & 1) * kMsgStride + kMsgL)[h];
        if (p.nsplit == 1) {
          const float inv = lr > 0.f ? 1.f / lr : 0.f;
          uint16_t* orow = p.out + (static_cast<int64_t>(row) * kHeads + h) * 512;
#pragma unroll 1
          for (int cc = 0; cc < 512 / 32; ++cc) {
            float o[32];
            tmem_ld32_sync(lane_base + 32 * cc, o);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 v;
              v.x = pack_bf16(o[j] * inv, o[j + 1] * inv);
              v.y = pack_bf16(o[j + 2] * inv, o[j + 3] * inv);
              v.z = pack_bf16(o[j + 4] * inv, o[j + 5] * inv);
              v.w = pack_bf16(o[j + 6] * inv, o[j + 7] * inv);
              *reinterpret_cast<uint4*>(orow + 32 * cc + j) = v;
            }
          }
        } else {
          // unnormalised partial O: columns [256 vh, 256 vh + 256) into block vh
#pragma unroll 1
          for (int cc = 0; cc < 512 / 32; ++cc) {
            float o[32];
            tmem_ld32_sync(lane_base + 32 * cc, o);
            float* orow = partial_block(p, row, cc >> 3, split) + h * kHalf + 32 * (cc & 7);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(orow + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
          }
        }
      }
    } else if (!bad && ntile == 0 && p.nsplit == 1) {
      uint16_t* orow = p.out + (static_cast<int64_t>(row) * kHeads + h) * 512;
      for (int j = 0; j < 512; j += 8)
        *reinterpret_cast<uint4*>(orow + j) = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merges the split partials: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// Grid (row, value half, head group of kCombineHeads); thread t owns output
// column t of the half for the group's heads, so the loads of all its heads
// are in flight together (a loop over the 128 heads with one dependent load
// each was latency-bound: ~60 us at 32 rows x 2 splits).
constexpr int kCombineHeads = 16;
__global__ void __launch_bounds__(256) mla_combine_kernel(const MParams p) {
  const int row = blockIdx.x;
  const int vh = blockIdx.y;
  const int h0 = blockIdx.z * kCombineHeads;
  const int t = threadIdx.x;
  pdl_launch_dependents_and_wait();
  const int64_t blk_floats = kHeads * kHalf + 2 * kHeads;
  const float* base = p.ws + (static_cast<int64_t>(row) * 2 + vh) * p.nsplit * blk_floats;
  __shared__ float wsh[64][kCombineHeads];  // nsplit <= 64
  __shared__ float inv_l[kCombineHeads];
  if (t < kCombineHeads) {
    const int h = h0 + t;
    float M = -INFINITY;
    for (int sp = 0; sp < p.nsplit; ++sp) M = fmaxf(M, base[sp * blk_floats + kHeads * kHalf + h]);
    float L = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) {
      const float m = base[sp * blk_floats + kHeads * kHalf + h];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      wsh[sp][t] = w;
      L += w * base[sp * blk_floats + kHeads * kHalf + kHeads + h];
    }
    inv_l[t] = L > 0.f ? 1.f / L : 0.f;
    if (vh == 0 && p.lse)
      p.lse[static_cast<int64_t>(row) * kHeads + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  float acc[kCombineHeads];
#pragma unroll
  for (int j = 0; j < kCombineHeads; ++j) acc[j] = 0.f;
  for (int sp = 0; sp < p.nsplit; ++sp) {
    const float* o = base + sp * blk_floats + static_cast<int64_t>(h0) * kHalf + t;
    float v[kCombineHeads];
#pragma unroll
    for (int j = 0; j < kCombineHeads; ++j) v[j] = o[j * kHalf];
    // a split with no valid selection has weight 0 and an unwritten O block:
    // its values are never used
#pragma unroll
    for (int j = 0; j < kCombineHeads; ++j) {
      const float w = wsh[sp][j];
      if (w != 0.f) acc[j] = fmaf(w, v[j], acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < kCombineHeads; ++j)
    p.out[(static_cast<int64_t>(row) * kHeads + h0 + j) * 512 + vh * kHalf + t] =
        __bfloat16_as_ushort(__float2bfloat16_rn(acc[j] * inv_l[j]));
}

// Splits of each row's selections: doubled while the CTA pairs of all rows
// and splits (2 R ns CTAs) still fit the device's SMs in one wave.
int choose_nsplit(int R, int k, int sm_count) {
  int ns = 1;
  const int max_split = (k + kTile - 1) / kTile;
  while (2 * R * ns * 2 <= sm_count && ns * 2 <= max_split && ns * 2 <= 64) ns *= 2;
  return ns;
}

}  // namespace

size_t mla_workspace_size(int R, int k, int sm_count) {
  const int ns = choose_nsplit(R, k, sm_count);
  if (ns == 1) return 0;
  return static_cast<size_t>(R) * 2 * ns * (kHeads * kHalf + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_sparse_mla(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int R = a.row_bt ? a.rows : a.num_req * a.next_n;
  const int ns = choose_nsplit(R, a.k, dev.sm_count);
  const int tiles = (a.k + kTile - 1) / kTile;
  const int tps = ((tiles + ns - 1) / ns) * kTile;
  MParams p;
  p.q = a.q;
  p.kv = reinterpret_cast<const uint8_t*>(a.kv);
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.num_pages = a.num_pages;
  p.next_n = a.next_n;
  p.row_bt = a.row_bt;
  p.bt_num_rows = a.bt_num_rows;
  p.idx = a.idx;
  p.k = a.k;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.nsplit = ns;
  p.tokens_per_split = tps;
  p.out = a.out;
  p.lse = a.lse;
  p.ws = static_cast<float*>(a.ws);
  p.err = dev.err_word;
  CUtensorMap tq;
  {
    // q as [R * 128 rows (row-major heads), 576] bf16; one box = a [128 x 64]
    // K-chunk of a row's Q, 128-byte swizzle
    char msg[160];
    const uint64_t dims[2] = {static_cast<uint64_t>(kDqk), static_cast<uint64_t>(R) * kHeads};
    const uint64_t strides[1] = {kDqk * 2};
    const uint32_t box[2] = {64, kHeads};
    if (!encode_tensor_map(&tq, 1, 2, const_cast<uint16_t*>(a.q), dims, strides, box, true, msg,
                           sizeof(msg)))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  // one cluster of two CTAs (score, value) per (row, split)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * R, ns, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, sparse_mla_kernel, tq, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || ns == 1) return e;
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(R, 2, kHeads / kCombineHeads);
  ccfg.blockDim = dim3(256);
  ccfg.stream = stream;
  ccfg.attrs = attr + 1;
  ccfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&ccfg, mla_combine_kernel, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

// ------------------------------------------------ no-allocation variant --
// Split-K scratch for callers that cannot allocate device memory.  The array
// lives in the module for as long as the library is loaded, once per device.
namespace {

constexpr size_t kStaticScratchBytes = size_t(24) << 20;  // 24 MiB
static __device__ __align__(256) unsigned char g_mla_static_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices] = {};

// Device address of this device's copy of the array.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
cudaError_t static_scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_mla_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = ptr;
  }
  *out = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace

size_t mla_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t launch_sparse_mla_static(const MlaArgs& a_in, const DeviceInfo& dev,
                                     cudaStream_t stream) {
  // The address is looked up on every call's first use of a device, split or
  // not, so a later call (perhaps under stream capture) makes no runtime query.
  void* ptr = nullptr;
  const cudaError_t e = static_scratch_address(dev.device, &ptr);
  if (e != cudaSuccess) return e;
  const int R = a_in.row_bt ? a_in.rows : a_in.num_req * a_in.next_n;
  const size_t need = mla_workspace_size(R, a_in.k, dev.sm_count);
  if (need > kStaticScratchBytes) return cudaErrorInvalidValue;  // the caller checks first
  MlaArgs a = a_in;
  a.ws = need > 0 ? ptr : nullptr;
  a.ws_bytes = need > 0 ? kStaticScratchBytes : 0;
  return launch_sparse_mla(a, dev, stream);
}

}  // namespace dsa
