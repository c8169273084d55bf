// Sparse MLA decode, Eq. (2) of "DeepSeek V3.2-Exp support" (llama.cpp issue
// 16331, section "1. Architecture"): attention of each query row's 128 heads
// over only the k selected latents c_s (576 = 512 latent + 64 rope elements;
// the value is the first 512).
//
// Work unit = one CTA per (row, value half vh, split); 128 selected tokens per
// tile.
//   warps 0-7  gather: Q of the row once (TMA, nine 128B-swizzled [128 x 64]
//              K-chunks); then per tile the nine [128 tokens x 64] K-chunks of
//              the selected latents, and one tile later the four value chunks
//              of this CTA's half again (an L2 hit), through a 5-slot ring of
//              16 KB, by 16-byte cp.async (each thread copies 4 pieces of a
//              chunk; completion is signalled with cp.async.mbarrier.arrive, so
//              no thread waits for its copies; a skipped selection is
//              zero-filled);
//   warps 8-11 softmax (one thread per head / TMEM lane): mask skipped
//              selections, running max with lazy rescaling of O (only when the
//              max grows by more than 2^8), P = exp2(S*scale*log2e - m) packed as
//              bf16 into the TMEM columns of the S tile it came from;
//   warp 12    tcgen05 issuer of S = Q K^T (kind::f16, M = 128 heads, N = 128
//              tokens, K = 576) into one of two TMEM tiles;
//   warp 13    tcgen05 issuer of O[128 x 256] += P V_half with P read from TMEM
//              and V read MN-major from the ring (N = 256 when the four value
//              chunks are contiguous in the ring, else two MMAs).  The ring
//              holds, in order, S(0), S(1), PV(0), S(2), PV(1), ...
// Many gathering warps matter: scattered 128-byte latent lines reach ~4-5 TB/s
// this way, about twice the rate of TMA tile::gather4 for the same lines.
// The 512 value columns are split over two CTAs because O for 128 heads x 512
// columns in f32 would fill all 512 TMEM columns; each CTA recomputes S.
// With more than one split the CTAs write unnormalised partial O plus their
// (max, sum) and a combine kernel merges them.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kThreads = 32 * (kGatherWarps + 4 + 2);  // gather, softmax, S MMA, PV MMA
constexpr int kMmaWarp = kGatherWarps + 4;
constexpr int kPvWarp = kMmaWarp + 1;
constexpr int kRing = 5;
constexpr int kTile = 128;
constexpr int kChunks = 9;  // 576 / 64
constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kHalf = 256;
constexpr int kTargetCtas = 152;
constexpr uint32_t kChunkBytes = kTile * 128;  // 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct MParams {
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

struct MSmem {
  uint8_t q[kChunks][kHeads * 128];  // 9 x 16 KB, K-major SW128, rows = heads
  uint8_t ring[kRing][kChunkBytes];  // [128 tokens x 64 elems] bf16 SW128
  uint64_t q_full;
  // a slot's use is signalled on full[] (an S chunk) or fullv[] (a value
  // chunk): each barrier has one consumer thread, which waits every phase
  // in order, so a parity wait cannot pass on an older phase
  uint64_t full[kRing], fullv[kRing], empty[kRing];
  uint64_t s_full[2];
  uint64_t p_full[2], pv_done[2];  // per S/P tile: tile t uses index t & 1
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }

// 2^x by the hardware approximation (a few ulp; P is rounded to bf16 anyway).
// 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const MParams p) {
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescS = make_idesc(1, 1, 128, kTile, false, false);
  constexpr int kSCol = 0;    // S/P tiles at columns [0, 256)
  constexpr int kOCol = 256;  // O half at columns [256, 512)
  extern __shared__ uint8_t smem_raw[];
  MSmem& s = *reinterpret_cast<MSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int row = blockIdx.x;
  const int vh = blockIdx.y;
  const int split = blockIdx.z;
  // the block-table row of this query row (an out-of-range one reads nothing)
  int req = p.row_bt ? p.row_bt[row] : row / p.next_n;
  if (p.row_bt && (req < 0 || req >= p.bt_num_rows)) {
    if (threadIdx.x == 0) raise_error(p.err, kErrBadPage);
    req = -1;
  }
  const int s0 = split * p.tokens_per_split;
  const int s1 = min(p.k, s0 + p.tokens_per_split);
  const int ntile = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(row) * p.k;

  if (tid == 0) {
    s.abort = 0;
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&s.full[i], 32 * kGatherWarps);  // one cp.async completion per gather thread
      mbar_init(&s.fullv[i], 32 * kGatherWarps);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.s_full[0], 1);
    mbar_init(&s.s_full[1], 1);
    // One arrival per softmax warp, one barrier per S/P tile: a warp can run one
    // tile ahead of the others (S(i+1) does not wait for P(i)), never two (S(i+2)
    // waits for PV(i)), so its arrival never lands in another tile's phase.
    mbar_init(&s.p_full[0], 4);
    mbar_init(&s.p_full[1], 4);
    // PV(t) commits to pv_done[t & 1].  With one barrier per tile parity every
    // waiter is within one phase of the phase it waits for (S(i) is issued only
    // after PV(i-2) completed), so a parity wait cannot alias an older phase.
    mbar_init(&s.pv_done[0], 1);
    mbar_init(&s.pv_done[1], 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile int* abort = &s.abort;

  if (warp < kGatherWarps) {
    // -------------------------------------------------------------- gather --
    const int gt = tid;  // 0 .. 32*kGatherWarps-1
    if (gt == 0 && ntile > 0) {
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(&s.q_full, kChunks * kHeads * 128);
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(s.q[c], &tm_q, &s.q_full, 64 * c, row * kHeads);
    }
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
          else if (pch == 0) raise_error(p.err, kErrBadIndex);
        }
      }
    };
    int tk_next[4], rows_cur[4], rows_prev[4] = {-1, -1, -1, -1};
    {
      int t0[4], pg0[4];
      load_toks(0, t0);
      load_pages(t0, pg0);
      make_rows(t0, pg0, rows_cur);
      load_toks(1, tk_next);
    }
    int g = 0;  // ring sequence number
    bool bad = false;
    auto issue = [&](int c, const int (&r)[4], bool value) -> bool {
      const int slot = g % kRing;
      if (g >= kRing && !mbar_wait_warp(&s.empty[slot], ((g / kRing) - 1) & 1, p.err, abort))
        return false;
      uint8_t* dst = s.ring[slot];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint8_t* d = dst + sw128_offset(prow + kRowStep * u, pch);
        if (r[u] >= 0)
          cp_async_16(d, p.kv + static_cast<int64_t>(r[u]) * (kDqk * 2) + c * 128 + pch * 16);
        else
          cp_async_16_zero(d, p.kv);
      }
      cp_async_mbar_arrive_noinc(value ? &s.fullv[slot] : &s.full[slot]);
      ++g;
      return true;
    };
    for (int i = 0; i <= ntile && !bad; ++i) {
      // loads for the next tiles go out first; their results are used after
      // this tile's copies have been issued
      int pg_next[4] = {-1, -1, -1, -1}, tk_after[4] = {-1, -1, -1, -1};
      if (i + 1 < ntile) {
        load_pages(tk_next, pg_next);
        load_toks(i + 2, tk_after);
      }
      if (i < ntile)
        for (int c = 0; c < kChunks && !bad; ++c) bad = !issue(c, rows_cur, false);
      if (i >= 1)
        for (int j = 0; j < 4 && !bad; ++j) bad = !issue(4 * vh + j, rows_prev, true);
      int rows_next[4] = {-1, -1, -1, -1};
      if (i + 1 < ntile) make_rows(tk_next, pg_next, rows_next);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        rows_prev[u] = rows_cur[u];
        rows_cur[u] = rows_next[u];
        tk_next[u] = tk_after[u];
      }
    }
    cp_async_wait<0>();  // no copy of this thread is left in flight at exit
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------- S MMA issuer --
    // One thread runs each MMA role: an M=128 MMA holds the issuing thread for
    // ~96-128 cycles, longer than the tensor core needs for it, so S (this
    // warp) and P V (the next warp) are issued by two threads.  Their MMAs
    // touch disjoint TMEM (S(i+1) its tile, PV(i) P(i) and O), and each
    // thread's commits track only its own MMAs.  Ring order: S(0), then per
    // tile i >= 1 S(i) followed by PV(i-1), and PV(ntile-1) last; S(i) starts
    // at ring sequence number 13 i - 4 (i >= 1).
    if (lane == 0 && ntile > 0 && mbar_wait(&s.q_full, 0, p.err, abort)) {
      uint32_t phase = 0;  // bit j: parity of the next phase of full[j]
      for (int i = 0; i < ntile && !*abort; ++i) {
        bool bad = false;
        int g = i == 0 ? 0 : (kChunks + 4) * i - 4;
        {
          const int buf = i & 1;
          // the S/P tile is reused after PV(i-2) has read P(i-2) from it
          if (i >= 2 && !mbar_wait(&s.pv_done[i & 1], ((i - 2) >> 1) & 1, p.err, abort)) break;
          tc_fence_after();
          const uint32_t dS = s.tmem_base + kSCol + buf * kTile;
          for (int c = 0; c < kChunks; ++c, ++g) {
            const int slot = g % kRing;
            if (!mbar_wait(&s.full[slot], (phase >> slot) & 1, p.err, abort)) { bad = true; break; }
            phase ^= 1u << slot;
            fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core
            tc_fence_after();
            const uint32_t a0 = smem_u32(s.q[c]);
            const uint32_t b0 = smem_u32(s.ring[slot]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(dS, sw128_desc(a0 + 32 * kk, 16, 1024), sw128_desc(b0 + 32 * kk, 16, 1024),
                      kIdescS, (c | kk) != 0);
            mma_commit(&s.empty[slot]);
          }
          if (bad) break;
          mma_commit(&s.s_full[buf]);
        }
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------- PV MMA issuer --
    // PV(t) reads ring sequence numbers 13 t + 18 .. (after S(t+1)), or
    // 13 t + 9 .. for the last tile.
    if (lane == 0 && ntile > 0) {
      uint32_t phase = 0;  // bit j: parity of the next phase of fullv[j]
      for (int t = 0; t < ntile && !*abort; ++t) {
        bool bad = false;
        const int g = t + 1 < ntile ? (kChunks + 4) * t + 18 : (kChunks + 4) * t + kChunks;
        {
          if (!mbar_wait(&s.p_full[t & 1], (t >> 1) & 1, p.err, abort)) break;
          for (int j = 0; j < 4 && !bad; ++j) {
            const int gg = g + j;
            const int slot = gg % kRing;
            bad = !mbar_wait(&s.fullv[slot], (phase >> slot) & 1, p.err, abort);
            phase ^= 1u << slot;
          }
          if (bad) break;
          fence_proxy_async_smem();
          tc_fence_after();
          // value chunk j sits in slot (g + j) % kRing: one or two contiguous runs
          const int first = g % kRing;
          const int n1 = min(4, kRing - first);  // chunks in the first run
          const uint32_t pa = s.tmem_base + kSCol + (t & 1) * kTile;
          const uint32_t v0 = smem_u32(s.ring[first]);
          const uint32_t v1 = smem_u32(s.ring[0]);
#pragma unroll 1
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
            mma_f16_ts(s.tmem_base + kOCol, pa + 8 * kk,
                       sw128_desc(v0 + 2048 * kk, kChunkBytes, 1024),
                       make_idesc(1, 1, 128, 64 * n1, false, true), acc);
            if (n1 < 4)
              mma_f16_ts(s.tmem_base + kOCol + 64 * n1, pa + 8 * kk,
                         sw128_desc(v1 + 2048 * kk, kChunkBytes, 1024),
                         make_idesc(1, 1, 128, 64 * (4 - n1), false, true), acc);
          }
          for (int j = 0; j < 4; ++j) mma_commit(&s.empty[(g + j) % kRing]);
          mma_commit(&s.pv_done[t & 1]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ softmax / epilogue --
    const int quad = warp & 3;  // warps 8-11: TMEM lane quadrants 0-3
    const int h = quad * 32 + lane;  // head == TMEM lane
    const uint32_t lane_base = s.tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool bad = false;
    // validity of a tile's 128 selections: lane j of every warp reads entries
    // j, 32+j, 64+j, 96+j; four ballots give the tile's mask (read a tile ahead)
    auto load_sel = [&](int i, int (&v)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = s0 + i * kTile + 32 * u + lane;
        v[u] = (i < ntile && pos < s1) ? idx_row[pos] : -1;
      }
    };
    int sel[4];
    load_sel(0, sel);
    for (int i = 0; i < ntile; ++i) {
      unsigned m[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) m[u] = __ballot_sync(0xffffffffu, sel[u] >= 0);
      load_sel(i + 1, sel);
      const bool all_valid = (m[0] & m[1] & m[2] & m[3]) == 0xffffffffu;  // warp-uniform
      const int buf = i & 1;
      if (!mbar_wait_warp(&s.s_full[buf], (i >> 1) & 1, p.err, abort)) { bad = true; break; }
      tc_fence_after();
      const uint32_t sbase = lane_base + kSCol + buf * kTile;
      // One pass over the tile's scores (log2 units, -inf if skipped), 64
      // columns at a time.  P = 2^(x - m_t) against the running reference m_t,
      // which only moves when a score exceeds it by more than the threshold
      // (then P already written for this tile is brought to the new m_t).
      // P is packed bf16 over the first 64 columns of this S tile: tokens
      // 0..63 -> columns 0..31 (their scores are read before anything is
      // written), then tokens 64..127 -> columns 32..63.
      float m_t = m_run, l_t = 0.f;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[64];
        tmem_ld64_sync(sbase + 64 * half, v);
        float h4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (all_valid) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            v[j] *= p.scale_log2;
            h4[j & 3] = fmaxf(h4[j & 3], v[j]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int t = 64 * half + j;
            const bool ok = ((m[t >> 5] >> (t & 31)) & 1u) != 0;
            v[j] = ok ? v[j] * p.scale_log2 : -INFINITY;
            h4[j & 3] = fmaxf(h4[j & 3], v[j]);
          }
        }
        const float hm = fmaxf(fmaxf(h4[0], h4[1]), fmaxf(h4[2], h4[3]));
        const bool grow = hm > m_t + kRescaleThreshold || (m_t == -INFINITY && hm > -INFINITY);
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? hm : m_t;
          if (half == 1) {
            // bring this tile's first 32 columns of P to the new reference
            const float f = (grow && m_t > -INFINITY) ? ex2_approx(m_t - m_new) : 1.f;
            float qf[32];
            tmem_ld32_sync(sbase, qf);
            uint32_t q[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const uint32_t w = __float_as_uint(qf[j]);
              q[j] = pack_bf16(bf16_lo(w) * f, bf16_hi(w) * f);
            }
            tmem_st32_sync(sbase, q);
            l_t *= f;
          }
          m_t = m_new;
        }
        // m_t is -inf only while every score seen is -inf: those give P = 0
        const float mref = m_t == -INFINITY ? 0.f : m_t;
        uint32_t pk[32];
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float e0 = ex2_approx(v[2 * j] - mref);
          const float e1 = ex2_approx(v[2 * j + 1] - mref);
          pk[j] = pack_bf16(e0, e1);
          l4[j & 3] += e0 + e1;  // the exact weights (P itself is rounded to bf16)
        }
        l_t += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        tmem_st32_sync(sbase + 32 * half, pk);
      }
      // O and l hold earlier tiles against m_run: bring them to m_t
      const bool moved = m_t != m_run && m_run > -INFINITY;
      const float corr = moved ? ex2_approx(m_run - m_t) : 1.f;
      if (__any_sync(0xffffffffu, moved)) {
        // O must hold PV(i-1) complete before it is rescaled
        if (!mbar_wait_warp(&s.pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, p.err, abort)) { bad = true; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < kHalf / 32; ++cc) {
          float o[32];
          tmem_ld32_sync(lane_base + kOCol + 32 * cc, o);
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(o[j] * corr);
          tmem_st32_sync(lane_base + kOCol + 32 * cc, r);
        }
      }
      l_run = l_run * corr + l_t;
      m_run = m_t;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.p_full[buf]);
    }
    // ---- epilogue: O half of this CTA ----
    if (!bad && ntile > 0 &&
        mbar_wait_warp(&s.pv_done[(ntile - 1) & 1], ((ntile - 1) >> 1) & 1, p.err, abort)) {
      tc_fence_after();
      if (p.nsplit == 1) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint16_t* orow = p.out + (static_cast<int64_t>(row) * kHeads + h) * 512 + vh * kHalf;
#pragma unroll 1
        for (int cc = 0; cc < kHalf / 32; ++cc) {
          float o[32];
          tmem_ld32_sync(lane_base + kOCol + 32 * cc, o);
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
        if (vh == 0 && p.lse)
          p.lse[static_cast<int64_t>(row) * kHeads + h] =
              l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      } else {
        // partial: [row][vh][split] blocks of (128 x 256 O, 128 m, 128 l)
        float* blk = p.ws + ((static_cast<int64_t>(row) * 2 + vh) * p.nsplit + split) *
                                (kHeads * kHalf + 2 * kHeads);
        float* orow = blk + h * kHalf;
#pragma unroll 1
        for (int cc = 0; cc < kHalf / 32; ++cc) {
          float o[32];
          tmem_ld32_sync(lane_base + kOCol + 32 * cc, o);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(orow + 32 * cc + j) =
                make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
        blk[kHeads * kHalf + h] = m_run;
        blk[kHeads * kHalf + kHeads + h] = l_run;
      }
    } else if (ntile == 0) {
      if (p.nsplit == 1) {
        uint16_t* orow = p.out + (static_cast<int64_t>(row) * kHeads + h) * 512 + vh * kHalf;
        for (int j = 0; j < kHalf; j += 8)
          *reinterpret_cast<uint4*>(orow + j) = make_uint4(0, 0, 0, 0);
        if (vh == 0 && p.lse) p.lse[static_cast<int64_t>(row) * kHeads + h] = -INFINITY;
      } else {
        float* blk = p.ws + ((static_cast<int64_t>(row) * 2 + vh) * p.nsplit + split) *
                                (kHeads * kHalf + 2 * kHeads);
        blk[kHeads * kHalf + h] = -INFINITY;
        blk[kHeads * kHalf + kHeads + h] = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(s.tmem_base, kTmemCols);
  }
}

// Merges the split partials: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(256) mla_combine_kernel(const MParams p) {
  const int row = blockIdx.x;
  const int vh = blockIdx.y;
  const int t = threadIdx.x;
  const int64_t blk_floats = kHeads * kHalf + 2 * kHeads;
  const float* base = p.ws + (static_cast<int64_t>(row) * 2 + vh) * p.nsplit * blk_floats;
  __shared__ float wsh[64][kHeads];  // nsplit <= 64
  __shared__ float inv_l[kHeads];
  if (t < kHeads) {
    float M = -INFINITY;
    for (int sp = 0; sp < p.nsplit; ++sp) M = fmaxf(M, base[sp * blk_floats + kHeads * kHalf + t]);
    float L = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) {
      const float m = base[sp * blk_floats + kHeads * kHalf + t];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      wsh[sp][t] = w;
      L += w * base[sp * blk_floats + kHeads * kHalf + kHeads + t];
    }
    inv_l[t] = L > 0.f ? 1.f / L : 0.f;
    if (vh == 0 && p.lse)
      p.lse[static_cast<int64_t>(row) * kHeads + t] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  for (int h = 0; h < kHeads; ++h) {
    float acc = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) {
      const float w = wsh[sp][h];
      if (w != 0.f) acc += w * base[sp * blk_floats + h * kHalf + t];
    }
    p.out[(static_cast<int64_t>(row) * kHeads + h) * 512 + vh * kHalf + t] =
        __bfloat16_as_ushort(__float2bfloat16_rn(acc * inv_l[h]));
  }
}

int choose_nsplit(int R, int k) {
  int ns = 1;
  const int max_split = (k + kTile - 1) / kTile;
  while (2 * R * ns * 2 <= kTargetCtas && ns * 2 <= max_split && ns * 2 <= 64) ns *= 2;
  return ns;
}

}  // namespace

size_t mla_workspace_size(int R, int k) {
  const int ns = choose_nsplit(R, k);
  if (ns == 1) return 0;
  return static_cast<size_t>(R) * 2 * ns * (kHeads * kHalf + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_sparse_mla(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int R = a.row_bt ? a.rows : a.num_req * a.next_n;
  const int ns = choose_nsplit(R, a.k);
  const int tiles = (a.k + kTile - 1) / kTile;
  const int tps = ((tiles + ns - 1) / ns) * kTile;
  CUtensorMap tq;
  char msg[128];
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kDqk), static_cast<uint64_t>(R) * kHeads};
    const uint64_t strides[1] = {kDqk * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tensor_map(&tq, 1, 2, const_cast<uint16_t*>(a.q), dims, strides, box, true, msg,
                           sizeof(msg)))
      return cudaErrorInvalidValue;
  }
  MParams p;
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
  const size_t smem = sizeof(MSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  sparse_mla_kernel<<<dim3(R, 2, ns), kThreads, smem, stream>>>(tq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || ns == 1) return e;
  mla_combine_kernel<<<dim3(R, 2), 256, 0, stream>>>(p);
  return cudaGetLastError();
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
                                     cudaStream_t stream, size_t* need) {
  const int R = a_in.row_bt ? a_in.rows : a_in.num_req * a_in.next_n;
  *need = mla_workspace_size(R, a_in.k);
  if (*need > kStaticScratchBytes) return cudaErrorMemoryAllocation;
  MlaArgs a = a_in;
  a.ws = nullptr;
  a.ws_bytes = 0;
  if (*need > 0) {
    void* ptr = nullptr;
    const cudaError_t e = static_scratch_address(dev.device, &ptr);
    if (e != cudaSuccess) return e;
    a.ws = ptr;
    a.ws_bytes = kStaticScratchBytes;
  }
  return launch_sparse_mla(a, dev, stream);
}

}  // namespace dsa
