// Lightning-indexer logits over a paged FP8 key cache, Eq. (1) of "DeepSeek
// V3.2-Exp support" (llama.cpp issue 16331, section "1. Architecture"):
//
//   logits[r, t] = s_t * sum_h (w[r,h] * sq[r,h]) * ReLU(q'[r,h] . k'_t)
//
// One persistent CTA per SM walks a contiguous range of work chunks
// (a chunk = up to kChunkTiles tiles of 128 tokens of one row group; a row
// group = up to 4 query rows of one request, which read the same keys).
//
//   warps 0-3   TMA producers, warp w filling the key stages s == w (mod 4)
//               (tile i of the CTA goes to stage i mod kStages): two 64-token
//               key pages per tile
//               (cp.async.bulk.tensor, 128-byte swizzle) + their 2 x 256 B
//               of per-token scales (cp.async.bulk).  Warp 0 also puts the
//               group's q (one 2-D TMA box of N = 64*rows rows) and w*sq
//               into a Q slot.  One issuing warp alone does not keep enough
//               page copies in flight to reach the HBM rate on GB300.
//   warps 4-5   tcgen05 issuers (one thread each, warp 4 + m taking the
//               tiles i == m (mod 2)): D[128 tokens, N] = K[128, 128] *
//               Q[N, 128]^T, four kind::f8f6f4 MMAs (K = 32 each) into one of
//               kAcc(G) TMEM accumulators (4 when 4*N columns fit in TMEM,
//               else 2).  The MMA of tile i waits for the epilogue of tile
//               i - kAcc, so more accumulators take the MMA -> epilogue
//               latency off the load path; an M=128 MMA holds the issuing
//               thread for ~96 cycles, so two issuers let one wait on its
//               barriers while the other feeds the tensor pipe.
//   warps 6-13  two epilogue warpgroups, warpgroup w draining the tiles
//               t == w (mod 2) (hence the accumulators a == w (mod 2)): each
//               thread owns one token (one TMEM lane) and reduces
//               sum_h w'_h * max(d_h, 0) per row, times s_t, and stores the
//               row's logit (consecutive threads -> consecutive tokens).
//
// Decode (1-2 rows per group) is bound by the HBM read of the key cache
// (132 B per token); a prefill chunk (4 rows per group, N = 256) is bound by
// the tensor pipe and the epilogue ALU.
//
// With a histogram output (decode, at most 2 rows per group) the epilogue
// also counts every logit it writes into a per-row histogram of its 12-bit
// order-key prefix, in shared memory, and when the CTA leaves a row group it
// adds the group's counts to the rows' histograms in global memory: the first
// pass of the top-k (where its cutoff lies) done on the logits while they are
// still in registers.
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kProducerWarps = 4;  // stage st is always filled by producer warp st % 4
constexpr int kMmaWarp = kProducerWarps;  // first MMA warp (also owns the TMEM allocation)
constexpr int kMmaWarps = 2;               // divides kAcc: an accumulator has one issuer
constexpr int kFirstEpiWarp = kMmaWarp + kMmaWarps;
constexpr int kThreads = 32 * (kFirstEpiWarp + 8);
// Key stages (a stage is held from its copy's issue until the epilogue has seen
// its MMAs complete).  Ten stages for up to two rows per group measured no
// faster than eight on GB300.
__host__ __device__ constexpr int stages_for(int) { return 8; }
constexpr int kTileTokens = 128;
constexpr uint32_t kPageKeyBytes = 64 * 128;  // 8192
constexpr uint32_t kStageBytes = 2 * kPageKeyBytes;
constexpr int kChunkTiles = 8;
constexpr int kMaxReq = 4096;

struct KParams {
  const float* q_scale;
  const float* w;
  const uint8_t* k_scale;
  int64_t s_page_stride;
  int num_pages;
  const int32_t* bt;
  int64_t bt_stride;
  const int32_t* ctx_len;
  int num_req;
  int next_n;               // rows per request, or (with cu_rows) at most this many
  const int32_t* cu_rows;   // null, or [num_req + 1]: request i's rows are [cu_rows[i], cu_rows[i+1])
  const int32_t* bt_rows;   // null, or [num_req]: the block-table row of request i
  int total_rows;           // with cu_rows: the rows of q and logits
  int bt_num_rows;          // with bt_rows: the rows of the block table
  float* logits;
  int64_t ld;
  uint32_t* hist;           // null, or [rows, kHistBins] (zero on entry; counts are added)
  uint32_t* err;
};

__device__ __forceinline__ int div_up(int a, int b) { return (a + b - 1) / b; }

// Rows of request i: next_n, or (varlen) cu_rows[i+1] - cu_rows[i]; a range
// outside [0, total_rows] is treated as empty (and reported by the caller).
__device__ __forceinline__ int rows_of(const int32_t* cu, int next_n, int total, int i) {
  if (!cu) return next_n;
  const int a = cu[i], b = cu[i + 1];
  return (a < 0 || b < a || b > total) ? 0 : b - a;
}
__device__ __forceinline__ bool bad_rows(const int32_t* cu, int total, int i) {
  return cu && (cu[i] < 0 || cu[i + 1] < cu[i] || cu[i + 1] > total);
}

__device__ __forceinline__ int group_tiles(int ctx, int next_n, int G, int gsub) {
  const int jlast = min(gsub * G + G, next_n) - 1;
  const int L = ctx - (next_n - 1 - jlast);
  return L <= 0 ? 0 : div_up(L, kTileTokens);
}

// Walks the chunks [c, c_end) of this CTA in order.  Every role runs an
// identical cursor, so they agree on the sequence of (group, tile range)
// without talking to each other.
struct Cursor {
  const int* prefix;  // smem [num_req + 1] exclusive chunk prefix per request
  const int32_t* ctx_len;
  const int32_t* cu_rows;  // null: every request has next_n rows
  int num_req, next_n, G, total_rows;
  int c, c_end;
  int req, gsub, ctx, tiles, gchunk, nchunk;
  int nn, ngroups, rbase;  // the current request's rows, row groups, first row
  int gcount;  // groups entered so far (the current group's Q slot is gcount & 1)

  __device__ void enter_request() {
    ctx = ctx_len[req];
    nn = rows_of(cu_rows, next_n, total_rows, req);
    rbase = cu_rows ? cu_rows[req] : req * next_n;
    ngroups = div_up(nn, G);
  }
  __device__ void enter_group() {
    tiles = group_tiles(ctx, nn, G, gsub);
    nchunk = div_up(tiles, kChunkTiles);
  }
  // Moves to the first group with chunks at or after (req, gsub).
  __device__ void settle() {
    for (;;) {
      if (req >= num_req) return;
      if (gsub >= ngroups || prefix[req + 1] == prefix[req]) {
        ++req;
        gsub = 0;
        if (req < num_req) enter_request();
        continue;
      }
      enter_group();
      if (nchunk > 0) return;
      ++gsub;
    }
  }
  __device__ void init(const int* pre, const int32_t* ctxs, const int32_t* cu, int total,
                       int nreq, int nrows_req, int g, int c0, int c1) {
    prefix = pre;
    ctx_len = ctxs;
    cu_rows = cu;
    total_rows = total;
    num_req = nreq;
    next_n = nrows_req;
    G = g;
    c = c0;
    c_end = c1;
    gcount = 0;
    if (c >= c_end) return;
    int lo = 0, hi = num_req;  // largest req with prefix[req] <= c
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= c) lo = mid; else hi = mid;
    }
    req = lo;
    enter_request();
    int rem = c - prefix[req];
    gsub = 0;
    for (;;) {
      enter_group();
      if (rem < nchunk) break;
      rem -= nchunk;
      ++gsub;
    }
    gchunk = rem;
  }
  __device__ bool valid() const { return c < c_end; }
  __device__ int tile_begin() const { return gchunk * kChunkTiles; }
  __device__ int tile_end() const { return min(tiles, gchunk * kChunkTiles + kChunkTiles); }
  __device__ int row0() const { return rbase + gsub * G; }
  __device__ int nrows() const { return min(G, nn - gsub * G); }
  // Advances to the next chunk; returns true if it leaves the current group.
  __device__ bool next() {
    ++c;
    if (c >= c_end) return true;
    if (++gchunk < nchunk) return false;
    gchunk = 0;
    ++gsub;
    settle();
    ++gcount;
    return true;
  }
  // Row length of row j of the current group.
  __device__ int row_len(int j) const {
    const int jj = gsub * G + j;
    return max(0, ctx - (nn - 1 - jj));
  }
};

template <int G, bool kHist>
struct Smem {
  static constexpr int N = 64 * G;
  static constexpr uint32_t kQBytes = N * 128;
  static constexpr int kStages = stages_for(G);
  uint8_t keys[kStages][kStageBytes];  // 1024-aligned stage tiles
  uint8_t q[2][kQBytes];
  float scales[kStages][kTileTokens];
  alignas(16) float wq[2][N];
  int prefix[kMaxReq + 1];
  uint64_t full[kStages], empty[kStages];
  uint64_t qfull[2], qempty[2];
  uint64_t tfull[4], tempty[4];
  uint32_t tmem_base;
  int abort;
  int scan_tmp[kThreads];
  uint32_t hist[kHist ? G * kHistBins : 1];  // this CTA's counts for the current row group
};

template <int G, bool kHist>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const KParams p) {
  constexpr int N = 64 * G;
  constexpr int kAcc = 4 * N <= 512 ? 4 : 2;
  static_assert(kAcc % kMmaWarps == 0, "an accumulator must have a single MMA issuer");
  constexpr uint32_t kTmemCols = (kAcc * N <= 128) ? 128 : (kAcc * N <= 256 ? 256 : 512);
  constexpr uint32_t kIdesc = make_idesc(0, 0, 128, N, false, false);
  using S = Smem<G, kHist>;
  constexpr int kStages = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // The barriers and TMEM are set up before the wait for the previous kernel
  // (no global memory is touched until the wait).
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 4);  // the 4 epilogue warps of the tile (after tfull, so the MMA is done)
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);  // the 4 warps of the warpgroup that drains accumulator i
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.qfull[i], 32);     // the 32 lanes of producer warp 0 (w*sq) + TMA bytes
      mbar_init(&s.qempty[i], kMmaWarps + 8); // MMA commits + 8 epilogue warps
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s.tmem_base, kTmemCols);
  pdl_launch_dependents_and_wait();

  // ---- per-request chunk counts and their exclusive prefix (all threads) ----
  for (int i = tid; i < p.num_req; i += kThreads) {
    const int ctx = p.ctx_len[i];
    const int nn = rows_of(p.cu_rows, p.next_n, p.total_rows, i);
    if (bad_rows(p.cu_rows, p.total_rows, i)) raise_error(p.err, kErrBadIndex);
    const int ngroups = nn > 0 ? div_up(nn, G) : 0;
    int n = 0;
    for (int g = 0; g < ngroups; ++g) n += div_up(group_tiles(ctx, nn, G, g), kChunkTiles);
    s.prefix[i + 1] = n;
  }
  if (tid == 0) {
    s.prefix[0] = 0;
    s.abort = 0;
  }
  if constexpr (kHist)
    for (int i = tid; i < G * kHistBins; i += kThreads) s.hist[i] = 0;
  __syncthreads();
  {
    // Each thread sums a contiguous segment; one warp scans the partials.
    const int n = p.num_req;
    const int seg = div_up(n, kThreads);
    const int a = min(n, tid * seg), b = min(n, a + seg);
    int sum = 0;
    for (int i = a; i < b; ++i) sum += s.prefix[i + 1];
    s.scan_tmp[tid] = sum;
    __syncthreads();
    if (warp == 0) {
      constexpr int per = kThreads / 32;
      int loc[per];
      int tot = 0;
#pragma unroll
      for (int i = 0; i < per; ++i) {
        loc[i] = s.scan_tmp[lane * per + i];
        tot += loc[i];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - tot;
#pragma unroll
      for (int i = 0; i < per; ++i) {
        s.scan_tmp[lane * per + i] = run;
        run += loc[i];
      }
    }
    __syncthreads();
    int run = s.scan_tmp[tid];
    for (int i = a; i < b; ++i) {
      run += s.prefix[i + 1];
      s.prefix[i + 1] = run;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = s.prefix[p.num_req];
  const int c0 = static_cast<int>((static_cast<long long>(total) * blockIdx.x) / gridDim.x);
  const int c1 = static_cast<int>((static_cast<long long>(total) * (blockIdx.x + 1)) / gridDim.x);
  volatile int* abort = &s.abort;

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers --
    Cursor cur;
    cur.init(s.prefix, p.ctx_len, p.cu_rows, p.total_rows, p.num_req, p.next_n, G, c0, c1);
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      if (warp == 0) tma_prefetch_desc(&tm_q);
    }
    // Decode (at most 2 rows per group) reads the key cache once per step: its
    // lines go first out of L2, which leaves the logits this kernel writes in
    // L2 for the top-k that reads them next.  A prefill chunk (4 rows per
    // group) reads the same keys once per row group: they stay in L2 instead.
    const uint64_t key_policy = G <= 2 ? l2_policy_evict_first() : l2_policy_evict_last();
    // Page ids of a chunk (at most 2 * kChunkTiles) are loaded by the lanes of
    // this warp one chunk ahead, so no block-table load sits on the TMA issue path.
    auto chunk_pages = [&](const Cursor& c) -> int {
      if (!c.valid()) return -1;
      const int npg = div_up(c.row_len(c.nrows() - 1), 64);
      const int pg = 2 * c.tile_begin() + lane;
      if (lane >= 2 * kChunkTiles || pg >= npg) return -1;
      const int64_t btr = p.bt_rows ? p.bt_rows[c.req] : c.req;
      if (btr < 0 || (p.bt_rows && btr >= p.bt_num_rows)) return -2;  // reported as a bad page
      return pg < p.bt_stride ? p.bt[btr * p.bt_stride + pg] : -2;
    };
    Cursor ahead = cur;
    int pages_cur = chunk_pages(cur);
    if (ahead.valid()) ahead.next();
    int pages_next = chunk_pages(ahead);
    int lt = 0;  // local tile counter
    int issued[kStages / kProducerWarps] = {};  // copies issued into this warp's stages
    int q_issued[2] = {0, 0};                   // warp 0: Q loads issued into each slot
    bool new_group = true;
    while (cur.valid() && !*abort) {
      const int r0 = cur.row0();
      const int nr = cur.nrows();
      if (new_group && warp == 0) {
        const int slot = cur.gcount & 1;
        const int use = cur.gcount >> 1;
        if (use > 0 && !mbar_wait_warp(&s.qempty[slot], (use - 1) & 1, p.err, abort)) break;
        for (int i = lane; i < N; i += 32) {
          const int j = i >> 6, h = i & 63;
          float v = 0.f;
          if (j < nr) v = p.w[(r0 + j) * 64 + h] * p.q_scale[(r0 + j) * 64 + h];
          s.wq[slot][i] = v;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.qfull[slot], S::kQBytes);
          tma_load_2d(s.q[slot], &tm_q, &s.qfull[slot], 0, r0 * 64);
        } else {
          mbar_arrive(&s.qfull[slot]);
        }
        ++q_issued[slot];
      }
      const int npages_grp = div_up(cur.row_len(nr - 1), 64);
      const int tb = cur.tile_begin();
      bool bad = false;
      for (int t = tb; t < cur.tile_end(); ++t, ++lt) {
        if ((lt % kStages) % kProducerWarps != warp) continue;
        const int st = lt % kStages;
        const int use = lt / kStages;
        if (use > 0 && !mbar_wait_warp(&s.empty[st], (use - 1) & 1, p.err, abort)) { bad = true; break; }
        const int pid0 = __shfl_sync(0xffffffffu, pages_cur, 2 * (t - tb));
        const int pid1 = __shfl_sync(0xffffffffu, pages_cur, 2 * (t - tb) + 1);
        ++issued[st / kProducerWarps];
        if (lane == 0) {
          const int pg1 = 2 * t + 1;
          const bool two = pg1 < npages_grp;
          mbar_arrive_expect_tx(&s.full[st], (two ? 2u : 1u) * (kPageKeyBytes + 256u));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1 && !two) break;
            int page = h ? pid1 : pid0;
            if (page < 0 || page >= p.num_pages) {
              raise_error(p.err, kErrBadPage);
              page = 0;
            }
            tma_load_3d_hint(s.keys[st] + h * kPageKeyBytes, &tm_k, &s.full[st], 0, 0, page,
                             key_policy);
            bulk_load_hint(&s.scales[st][h * 64],
                           p.k_scale + static_cast<int64_t>(page) * p.s_page_stride, 256,
                           &s.full[st], key_policy);
          }
        }
        __syncwarp();
      }
      if (bad) break;
      new_group = cur.next();
      pages_cur = pages_next;
      if (ahead.valid()) {
        ahead.next();
        pages_next = chunk_pages(ahead);
      }
    }
    // every copy this warp issued has landed before the CTA can exit (at once
    // unless a wait ran out and the consumers stopped early)
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kStages / kProducerWarps; ++i)
        if (issued[i] > 0) mbar_drain(&s.full[warp + kProducerWarps * i], (issued[i] - 1) & 1, p.err);
      for (int i = 0; i < 2; ++i)
        if (q_issued[i] > 0) mbar_drain(&s.qfull[i], (q_issued[i] - 1) & 1, p.err);
    }
    __syncwarp();
  } else if (warp < kFirstEpiWarp) {
    // ---------------------------------------------------------- MMA issuers --
    // One thread per MMA warp: the per-tile loop is on the critical path of the
    // pipeline, so it carries no warp votes or warp barriers.
    const int m = warp - kMmaWarp;
    if (lane == 0) {
      Cursor cur;
      cur.init(s.prefix, p.ctx_len, p.cu_rows, p.total_rows, p.num_req, p.next_n, G, c0, c1);
      int lt = 0;
      bool new_group = true;
      while (cur.valid() && !*abort) {
        const int slot = cur.gcount & 1;
        if (new_group && !mbar_wait(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) break;
        const int tb = cur.tile_begin(), te = cur.tile_end();
        bool bad = false;
        const uint32_t b0 = smem_u32(s.q[slot]);
        for (int t = tb; t < te; ++t, ++lt) {
          if (lt % kMmaWarps != m) continue;
          const int st = lt % kStages;
          const int buf = lt % kAcc;
          const int ub = lt / kAcc;
          if (!mbar_wait(&s.full[st], (lt / kStages) & 1, p.err, abort)) { bad = true; break; }
          if (ub > 0 && !mbar_wait(&s.tempty[buf], (ub - 1) & 1, p.err, abort)) { bad = true; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(s.keys[st]);
          const uint32_t d = s.tmem_base + static_cast<uint32_t>(buf * N);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8f6f4(d, sw128_desc(a0 + 32 * k, 16, 1024), sw128_desc(b0 + 32 * k, 16, 1024),
                       kIdesc, k > 0);
          // completion of these MMAs also frees the key stage: the epilogue
          // releases it after it has seen tfull
          mma_commit(&s.tfull[buf]);
        }
        if (bad) break;
        new_group = cur.next();
        if (new_group) mma_commit(&s.qempty[slot]);
      }
    }
    __syncwarp();
  } else if constexpr (!kHist) {
    // ------------------------------------------------------------- epilogue --
    const int wg = (warp - kFirstEpiWarp) >> 2;  // which tiles (and accumulators) it drains
    const int quad = warp & 3;       // TMEM lane quadrant of this warp
    const int row_in_tile = quad * 32 + lane;
    Cursor cur;
    cur.init(s.prefix, p.ctx_len, p.cu_rows, p.total_rows, p.num_req, p.next_n, G, c0, c1);
    int lt = 0;
    while (cur.valid() && !*abort) {
      const int slot = cur.gcount & 1;
      bool waited_q = false;
      const int r0 = cur.row0();
      const int nr = cur.nrows();
      bool bad = false;
      for (int t = cur.tile_begin(); t < cur.tile_end(); ++t, ++lt) {
        if ((lt & 1) != wg) continue;
        if (!waited_q) {
          if (!mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) { bad = true; break; }
          waited_q = true;
        }
        const int st = lt % kStages;
        const int buf = lt % kAcc;
        if (!mbar_wait_warp(&s.tfull[buf], (lt / kAcc) & 1, p.err, abort)) { bad = true; break; }
        tc_fence_after();
        // the MMA has read the stage's keys (tfull); once every lane holds its
        // scale the stage can be refilled
        const float sc = s.scales[st][row_in_tile];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[st]);
        const int tok = t * kTileTokens + row_in_tile;
        const uint32_t taddr = s.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               static_cast<uint32_t>(buf * N);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float v[64];
          tmem_ld64_sync(taddr + j * 64, v);
          const float acc = relu_dot64(v, s.wq[slot] + j * 64);
          if (j < nr && tok < cur.row_len(j) && tok < p.ld)
            p.logits[static_cast<int64_t>(r0 + j) * p.ld + tok] = acc * sc;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.tempty[buf]);
      }
      if (bad) break;
      // A warp may walk through a group without processing any of its tiles (they
      // went to the other warpgroup).  It still waits for that group's Q before it
      // arrives on the slot's qempty, so its arrival cannot land in the phase of
      // the group that used the slot two groups earlier.
      if (!waited_q && !mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) break;
      const int gslot = slot;
      const bool left = cur.next();
      if (left && lane == 0) mbar_arrive(&s.qempty[gslot]);
      __syncwarp();
    }
  } else {
    // ------------------------------------- epilogue with score histograms --
    // A warp that has given up (a wait ran out) keeps walking the cursor
    // without doing work, so that it still meets the other epilogue warps at
    // every row-group barrier of the histogram flush.
    const int wg = (warp - kFirstEpiWarp) >> 2;  // which tiles (and accumulators) it drains
    const int quad = warp & 3;       // TMEM lane quadrant of this warp
    const int row_in_tile = quad * 32 + lane;
    const int etid = tid - 32 * kFirstEpiWarp;  // 0 .. 255
    Cursor cur;
    cur.init(s.prefix, p.ctx_len, p.cu_rows, p.total_rows, p.num_req, p.next_n, G, c0, c1);
    int lt = 0;
    bool bad = false;
    while (cur.valid()) {
      const int slot = cur.gcount & 1;
      bool waited_q = false;
      const int r0 = cur.row0();
      const int nr = cur.nrows();
      for (int t = cur.tile_begin(); t < cur.tile_end(); ++t, ++lt) {
        if ((lt & 1) != wg || bad) continue;
        if (!waited_q) {
          if (!mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) { bad = true; continue; }
          waited_q = true;
        }
        const int st = lt % kStages;
        const int buf = lt % kAcc;
        if (!mbar_wait_warp(&s.tfull[buf], (lt / kAcc) & 1, p.err, abort)) { bad = true; continue; }
        tc_fence_after();
        // the MMA has read the stage's keys (tfull); once every lane holds its
        // scale the stage can be refilled
        const float sc = s.scales[st][row_in_tile];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[st]);
        const int tok = t * kTileTokens + row_in_tile;
        const uint32_t taddr = s.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               static_cast<uint32_t>(buf * N);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float v[64];
          tmem_ld64_sync(taddr + j * 64, v);
          const float acc = relu_dot64(v, s.wq[slot] + j * 64);
          if (j < nr && tok < cur.row_len(j) && tok < p.ld) {
            const float logit = acc * sc;
            p.logits[static_cast<int64_t>(r0 + j) * p.ld + tok] = logit;
            atomicAdd(&s.hist[j * kHistBins + (order_key(logit) >> kHistShift)], 1u);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.tempty[buf]);
      }
      // A warp may walk through a group without processing any of its tiles (they
      // went to the other warpgroup).  It still waits for that group's Q before it
      // arrives on the slot's qempty, so its arrival cannot land in the phase of
      // the group that used the slot two groups earlier.
      if (!bad && !waited_q && !mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort))
        bad = true;
      const int gslot = slot;
      const bool left = cur.next();
      if (left && lane == 0 && !bad) mbar_arrive(&s.qempty[gslot]);
      __syncwarp();
      {
        if (left) {
          // both epilogue warpgroups are done with the group's tiles: add this
          // CTA's counts to the rows' global histograms and clear them
          const bool any_bad = named_bar_or(1, 256, bad);
          if (!any_bad) {
            for (int i = etid; i < nr * kHistBins; i += 256) {
              const uint32_t c = s.hist[i];
              if (c) {
                atomicAdd(&p.hist[static_cast<int64_t>(r0 + (i >> kHistBits)) * kHistBins +
                                  (i & (kHistBins - 1))],
                          c);
                s.hist[i] = 0;
              }
            }
          }
          named_bar_sync(1, 256);
          bad = bad || any_bad;
        }
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

template <int G, bool kHist>
cudaError_t launch_g(const IndexerArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                     const CUtensorMap& tk, const CUtensorMap& tq) {
  static_assert(sizeof(Smem<G, kHist>) + 1024 <= 227 * 1024, "indexer shared memory exceeds 227 KB");
  const size_t smem = sizeof(Smem<G, kHist>) + 1024;
  auto fn = indexer_kernel<G, kHist>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  KParams p;
  p.q_scale = a.q_scale;
  p.w = a.w;
  p.k_scale = a.k_scale;
  p.s_page_stride = a.s_page_stride;
  p.num_pages = a.num_pages;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.ctx_len = a.ctx_len;
  p.num_req = a.num_req;
  p.next_n = a.next_n;
  p.cu_rows = a.cu_rows;
  p.bt_rows = a.bt_rows;
  p.total_rows = a.total_rows;
  p.bt_num_rows = a.bt_num_rows;
  p.logits = a.logits;
  p.ld = a.ld;
  p.hist = a.hist;
  p.err = dev.err_word;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, tk, tq, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

cudaError_t launch_indexer(const IndexerArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                           char* msg, size_t msg_len) {
  if (a.num_req > kMaxReq) {
    snprintf(msg, msg_len, "dsa_indexer_logits: num_req %d exceeds %d", a.num_req, kMaxReq);
    return cudaErrorInvalidValue;
  }
  const int G = a.next_n >= 4 ? 4 : a.next_n;
  CUtensorMap tk, tq;
  {
    // keys: [num_pages][64 tokens][128 bytes], page stride k_page_stride
    const uint64_t dims[3] = {128, 64, static_cast<uint64_t>(a.num_pages)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(a.k_page_stride)};
    const uint32_t box[3] = {128, 64, 1};
    if (!encode_tensor_map(&tk, 0, 3, const_cast<uint8_t*>(a.k_cache), dims, strides, box, true,
                           msg, msg_len))
      return cudaErrorInvalidValue;
  }
  {
    // q: [R*64 rows][128 bytes]; one box = the N rows of a row group
    const uint64_t rows =
        (a.cu_rows ? static_cast<uint64_t>(a.total_rows) : static_cast<uint64_t>(a.num_req) * a.next_n) * 64;
    const uint64_t dims[2] = {128, rows};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {128, static_cast<uint32_t>(64 * G)};
    if (!encode_tensor_map(&tq, 0, 2, const_cast<uint8_t*>(a.q), dims, strides, box, true, msg,
                           msg_len))
      return cudaErrorInvalidValue;
  }
  if (a.hist) {
    if (G > 2) {
      snprintf(msg, msg_len, "score histograms need at most 2 query rows per request (next_n %d)",
               a.next_n);
      return cudaErrorInvalidValue;
    }
    return G == 1 ? launch_g<1, true>(a, dev, stream, tk, tq) : launch_g<2, true>(a, dev, stream, tk, tq);
  }
  switch (G) {
    case 1: return launch_g<1, false>(a, dev, stream, tk, tq);
    case 2: return launch_g<2, false>(a, dev, stream, tk, tq);
    case 3: return launch_g<3, false>(a, dev, stream, tk, tq);
    default: return launch_g<4, false>(a, dev, stream, tk, tq);
  }
}

}  // namespace dsa
