// Two-level candidate-block indexer (the vLLM "sparse_indexer" backend page:
// candidate consumer layers score only the candidate blocks published by the
// source layer; the first consumer of a step fills sparse_indices, end and the
// kernel schedule, later consumers reuse them; keys are MXFP4 with UE8M0
// scales at granularity 32).
//
// candidate_expand: one CTA per row sorts its block ids (bitonic sort in
// shared memory), counts the valid sparse columns (end) and writes the row's
// work-chunk count; a one-CTA scan turns the counts into the schedule (an
// exclusive prefix over rows) that candidate_logits walks.
//
// candidate_logits: the indexer pipeline of indexer.cu over candidate
// columns.  A tile is 128 sparse columns = two candidate blocks = two 64-token
// pages.  The keys stay e2m1 all the way to the tensor core: a TMA tensor copy
// whose element type is the 4-bit "16 values in 8 bytes, every 8 bytes padded
// to 16" form writes each page's 64 keys into the 128B-swizzled shared-memory
// layout in which the block-scaled kind::mxf8f6f4 MMA reads e2m1 operands
// (one element per byte of footprint), and a bulk copy brings the page's 64 x 4
// UE8M0 scale bytes.  Scale warps put each token's scale word into a
// tensor-memory scale block; an MMA issuer issues four block-scaled MMAs (A =
// keys e2m1, B = q e4m3, K = 32 each, group g taking byte g of the token's
// scale word, the q side scaled by 2^0) into one accumulator, so the tensor
// core applies the scales:
//   logit = sum_h w'_h * ReLU(sum_g 2^(e_g - 127) * (k_g . q'_g)[h]),
// and the epilogue is the dense indexer's (one accumulator, ReLU, weights).
#include <cuda_bf16.h>

#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

// Roles, each sized by measurement on GB300 (64 rows x 32768 columns per
// layer: one producer warp, one issuer and one epilogue warpgroup 69.9 us;
// 3 producers, 2 issuers and 2 epilogue warpgroups 55 us; 4 and 4 54 us: a
// warp's copies, and a lone issuing thread, are slow enough to set the pace):
//   warps 0-3   producers: warp w fills the stages of tiles == w (mod 4)
//   warps 4-7   MMA issuers: warp 4 + i issues the tiles == i (mod 4)
//   warps 8-11  scale warps (one per TMEM lane quadrant)
//   warps 12-19 two epilogue warpgroups: group g drains the tiles == g (mod 2)
constexpr int kProducers = 4;
constexpr int kMmaWarp = kProducers;
constexpr int kIssuers = 4;
constexpr int kScaleWarp = kMmaWarp + kIssuers;
constexpr int kFirstEpiWarp = kScaleWarp + 4;
constexpr int kThreads = 32 * (kFirstEpiWarp + 8);
constexpr int kStages = 12;  // key + scale stages
constexpr int kAcc = 4;      // [128 x 64] accumulators
// a stage is always filled by the same producer and issued by the same MMA
// thread, and an accumulator always drained by the same epilogue group, so no
// waiter ever looks at a barrier two phases ahead of it
static_assert(kStages % kProducers == 0 && kStages % kIssuers == 0 && kAcc % 2 == 0 &&
                  kAcc % kIssuers == 0,
              "role / ring sizes");
// Tensor-memory columns: the accumulators, then a 4-column scale block per
// stage (row m of the tile: column m / 32, lane m % 32 in every lane quadrant,
// byte g = the scale of its group g), then the q side's scale block (every
// byte 2^0); each block 16-column aligned.
constexpr uint32_t kSfaCol = 64 * kAcc;
constexpr uint32_t kSfStride = 16;
constexpr uint32_t kSfbCol = kSfaCol + kSfStride * kStages;
constexpr uint32_t kOneScales = 0x7F7F7F7Fu;  // four UE8M0 bytes of 2^0
constexpr uint32_t kFmtE2M1 = 5;              // instruction-descriptor code of e2m1
constexpr uint32_t kKeyPageSmem = 64 * 128;   // a page's keys in shared memory (padded e2m1)
// The tensor copy of 4-bit values completes its mbarrier transaction with the
// packed byte count read from global memory (measured on GB300), not with the
// padded bytes it writes.
constexpr uint32_t kKeyPageTx = 64 * 64;
constexpr int kTileCols = 128;
constexpr int kChunkTiles = 4;
constexpr uint32_t kSfPage = 64 * 4;  // a page's UE8M0 bytes

__device__ __forceinline__ int div_up(int a, int b) { return (a + b - 1) / b; }

// The row holding chunk c (sched[row] <= c < sched[row + 1]; sched is the
// exclusive prefix of the rows' chunk counts, sched[R] > c), found by one
// warp: each round the 32 lanes probe 32 evenly spaced rows, so R rows take
// ceil(log32 R) dependent loads instead of log2 R.
__device__ int find_row(const int32_t* sched, int R, int c) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = R;  // sched[lo] <= c < sched[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && sched[idx] <= c;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int j = 31 - __clz(m);  // lane 0 always qualifies (sched[lo] <= c)
    lo = lo + j * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

// ------------------------------------------------------------- expansion --

__global__ void __launch_bounds__(256) candidate_expand_kernel(CandExpandArgs a, uint32_t* err) {
  __shared__ int ids[4096];
  __shared__ int red[8];
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  int n2 = 1;
  while (n2 < a.nb) n2 <<= 1;
  // candidate block b covers the sparse blocks b*expand .. b*expand+expand-1;
  // ids past int32 range stay past the context (they sort last)
  const int m = a.expand;
  const int32_t* src = a.cand + static_cast<int64_t>(r) * (a.nb / m);
  for (int i = tid; i < n2; i += 256) {
    int v = 0x7fffffff;
    if (i < a.nb) {
      const int64_t b = static_cast<int64_t>(src[i / m]) * m + i % m;
      v = b > 0x7ffffffell ? 0x7fffffff : static_cast<int>(b);
    }
    ids[i] = v;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n2 / 2; i += 256) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const int x = ids[lo], y = ids[hi];
        if ((x > y) == asc) {
          ids[lo] = y;
          ids[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  const int req = r / a.next_n;
  const int j = r % a.next_n;
  const int64_t L = static_cast<int64_t>(a.ctx_len[req]) - (a.next_n - 1 - j);
  int cnt = 0;
  for (int i = tid; i < a.nb; i += 256) {
    const int b = ids[i];
    a.sparse_indices[static_cast<int64_t>(r) * a.nb + i] = b;
    if (b < 0) {
      raise_error(err, kErrBadIndex);
      continue;
    }
    const int64_t v = L - static_cast<int64_t>(b) * a.bs;
    cnt += static_cast<int>(v <= 0 ? 0 : (v >= a.bs ? a.bs : v));
  }
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) red[tid >> 5] = cnt;
  __syncthreads();
  if (tid == 0) {
    int tot = 0;
    for (int w = 0; w < 8; ++w) tot += red[w];
    a.end[r] = tot;
    int32_t* sched = static_cast<int32_t*>(a.schedule);
    sched[r + 1] = div_up(div_up(tot, kTileCols), kChunkTiles);
  }
}

// In-place exclusive prefix of sched[1..R] (sched[0] = 0) by one CTA.
__global__ void __launch_bounds__(1024) schedule_scan_kernel(int32_t* sched, int R) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    carry = 0;
    sched[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < R; base += 1024) {
    const int i = base + tid;
    int v = i < R ? sched[i + 1] : 0;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      int s = warp_sums[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    const int before = (w > 0 ? warp_sums[w - 1] : 0) + carry;
    if (i < R) sched[i + 1] = before + incl;
    __syncthreads();
    if (tid == 1023) carry = before + incl;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- logits --

struct CParams {
  const float* q_scale;
  const float* w;
  const uint8_t* k_fp4;
  int64_t k_page_stride;
  const uint8_t* k_sf;
  int64_t sf_page_stride;
  int num_pages;
  const int32_t* bt;
  int64_t bt_stride;
  int next_n;
  int R;
  const int32_t* sparse_indices;
  int nb;
  const int32_t* end;
  const int32_t* sched;  // [R+1] exclusive chunk prefix
  float* logits;          // f32 output, or
  uint16_t* logits_bf16;  // bf16 output (round to nearest even) when not null
  int64_t ld;
  uint32_t* err;
};

// Walks the chunks [c, c_end) of this CTA; one row per group.
struct RowCursor {
  const int32_t* sched;
  const int32_t* end;
  int R;
  int c, c_end, row, tiles, gchunk, nchunk, gcount;
  int max_cols;
  __device__ void enter() {
    tiles = div_up(min(end[row], max_cols), kTileCols);
    nchunk = div_up(tiles, kChunkTiles);
  }
  // row0: the row of chunk c0 (find_row), or anything when c0 >= c1
  __device__ void init(const int32_t* sc, const int32_t* en, int nrows, int c0, int c1,
                       int cols, int row0) {
    max_cols = cols;
    sched = sc;
    end = en;
    R = nrows;
    c = c0;
    c_end = c1;
    gcount = 0;
    if (c >= c_end) return;
    row = row0;
    enter();
    gchunk = c - sched[row];
  }
  __device__ bool valid() const { return c < c_end; }
  __device__ int tile_begin() const { return gchunk * kChunkTiles; }
  __device__ int tile_end() const { return min(tiles, gchunk * kChunkTiles + kChunkTiles); }
  __device__ bool next() {
    ++c;
    if (c >= c_end) return true;
    if (++gchunk < nchunk) return false;
    gchunk = 0;
    do {
      ++row;
    } while (row < R && sched[row + 1] == sched[row]);
    if (row < R) enter();
    ++gcount;
    return true;
  }
};

struct CSmem {
  uint8_t a[kStages][2 * kKeyPageSmem];  // a tile's keys, e2m1 padded, K-major SW128
  uint8_t q[2][64 * 128];                // q of the row, K-major SW128
  uint8_t sf[kStages][2 * kSfPage];      // a tile's 128 x 4 UE8M0 bytes
  alignas(16) float wq[2][64];
  uint64_t full[kStages], empty[kStages], sready[kStages];
  uint64_t qfull[2], qempty[2];
  uint64_t tfull[kAcc], tempty[kAcc];
  uint32_t tmem_base;
  int abort;
  int row0;  // the row of this CTA's first chunk
};

static_assert(sizeof(CSmem) + 1024 <= 227 * 1024, "candidate shared memory exceeds 227 KB");

__global__ void __launch_bounds__(kThreads, 1)
    candidate_logits_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k, const CParams p) {
  constexpr uint32_t kTmemCols = 512;  // accumulators + scale columns, rounded up to a power of 2
  static_assert(kSfbCol + 4 <= kTmemCols, "tensor-memory columns");
  extern __shared__ uint8_t smem_raw[];
  CSmem& s = *reinterpret_cast<CSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    s.abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);   // the MMA commit
      mbar_init(&s.sready[i], 4);  // the 4 scale warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.qfull[i], 32);
      mbar_init(&s.qempty[i], kIssuers + 8);  // the MMA issuers' commits + the 8 epilogue warps
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);  // the 4 epilogue warps
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the q side's scale block: every byte 2^0, in all 128 lanes (the four
  // epilogue warps cover the four lane quadrants)
  if (warp >= kFirstEpiWarp)
    tmem_st4_sync(s.tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kSfbCol,
                  kOneScales, kOneScales, kOneScales, kOneScales);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = p.sched[p.R];
  const int c0 = static_cast<int>((static_cast<long long>(total) * blockIdx.x) / gridDim.x);
  const int c1 = static_cast<int>((static_cast<long long>(total) * (blockIdx.x + 1)) / gridDim.x);
  volatile int* abort = &s.abort;
  if (warp == 0 && c0 < c1) {
    const int r = find_row(p.sched, p.R, c0);
    if (lane == 0) s.row0 = r;
  }
  __syncthreads();
  const int row0 = s.row0;

  if (warp < kProducers) {
    // ------------------------------------------------------------ producers --
    const int pw = warp;  // fills the stages of tiles == pw (mod kProducers)
    RowCursor cur;
    cur.init(p.sched, p.end, p.R, c0, c1, p.nb * 64, row0);
    if (pw == 0 && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
    }
    // The page of a tile column block takes two dependent loads (sparse
    // index, then block table).  Lane l holds block 2*tile_begin + l of a
    // chunk: its sparse index is loaded two chunks ahead and its page one chunk
    // ahead, so no load sits on the copy issue path.
    auto load_blk = [&](const RowCursor& c) -> int {
      if (!c.valid() || lane >= 2 * kChunkTiles) return -1;
      const int b = 2 * c.tile_begin() + lane;
      return b < p.nb ? p.sparse_indices[static_cast<int64_t>(c.row) * p.nb + b] : -1;
    };
    auto load_page = [&](const RowCursor& c, int blk) -> int {
      if (!c.valid() || lane >= 2 * kChunkTiles) return -1;
      if (blk < 0 || blk >= p.bt_stride) return -2;
      return p.bt[static_cast<int64_t>(c.row / p.next_n) * p.bt_stride + blk];
    };
    // keys are read once per layer: their lines go first out of L2, which
    // leaves the logits written here in L2 for the top-k that reads them next
    const uint64_t evict_first = l2_policy_evict_first();
    RowCursor ahead1 = cur, ahead2 = cur;
    int pages_cur = load_page(cur, load_blk(cur));
    if (ahead1.valid()) ahead1.next();
    int blk1 = load_blk(ahead1);
    ahead2 = ahead1;
    if (ahead2.valid()) ahead2.next();
    int blk2 = load_blk(ahead2);
    int pages1 = load_page(ahead1, blk1);
    int lt = 0, endr = 0;
    int q_issued[2] = {0, 0};  // Q loads issued into each slot (producer 0)
    int last_use[kStages / kProducers];  // phases issued into this producer's stages
#pragma unroll
    for (int i = 0; i < kStages / kProducers; ++i) last_use[i] = 0;
    bool new_group = true;
    while (cur.valid() && !*abort) {
      const int r = cur.row;
      if (new_group && pw == 0) {
        const int slot = cur.gcount & 1;
        const int use = cur.gcount >> 1;
        if (use > 0 && !mbar_wait_warp(&s.qempty[slot], (use - 1) & 1, p.err, abort)) break;
        for (int i = lane; i < 64; i += 32) s.wq[slot][i] = p.w[r * 64 + i] * p.q_scale[r * 64 + i];
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.qfull[slot], 64 * 128);
          tma_load_2d(s.q[slot], &tm_q, &s.qfull[slot], 0, r * 64);
        } else {
          mbar_arrive(&s.qfull[slot]);
        }
        ++q_issued[slot];
      }
      if (new_group) endr = min(p.end[r], p.nb * 64);
      const int tb = cur.tile_begin();
      bool bad = false;
      for (int t = tb; t < cur.tile_end(); ++t, ++lt) {
        if (lt % kProducers != pw) continue;
        const int st = lt % kStages;
        const int use = lt / kStages;
        if (use > 0 && !mbar_wait_warp(&s.empty[st], (use - 1) & 1, p.err, abort)) { bad = true; break; }
        last_use[st / kProducers] = use + 1;
        int pid[2];
        pid[0] = __shfl_sync(0xffffffffu, pages_cur, 2 * (t - tb));
        pid[1] = __shfl_sync(0xffffffffu, pages_cur, 2 * (t - tb) + 1);
        const bool two = (2 * t + 1) * 64 < endr;
        if (lane == 0)
          mbar_arrive_expect_tx(&s.full[st], (two ? 2u : 1u) * (kKeyPageTx + kSfPage));
        __syncwarp();
        // the tile's copies go out from different lanes
        if (lane < 4) {
          const int h = lane >> 1;  // which page of the tile
          if (h == 0 || two) {
            int page = pid[h];
            if (page < 0 || page >= p.num_pages) {
              if ((lane & 1) == 0) raise_error(p.err, kErrBadPage);
              page = 0;
            }
            if ((lane & 1) == 0)
              tma_load_3d_hint(s.a[st] + h * kKeyPageSmem, &tm_k, &s.full[st], 0, 0, page,
                               evict_first);
            else
              bulk_load_hint(s.sf[st] + h * kSfPage,
                             p.k_sf + static_cast<int64_t>(page) * p.sf_page_stride, kSfPage,
                             &s.full[st], evict_first);
          }
        }
        __syncwarp();
      }
      if (bad) break;
      new_group = cur.next();
      pages_cur = pages1;
      ahead1 = ahead2;
      blk1 = blk2;
      if (ahead2.valid()) ahead2.next();
      blk2 = load_blk(ahead2);
      pages1 = load_page(ahead1, blk1);
    }
    // every copy issued has landed before the CTA can exit (at once unless a
    // wait ran out and the consumers stopped early)
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kStages / kProducers; ++i)
        if (last_use[i] > 0) mbar_drain(&s.full[kProducers * i + pw], (last_use[i] - 1) & 1, p.err);
      for (int i = 0; i < 2; ++i)
        if (q_issued[i] > 0) mbar_drain(&s.qfull[i], (q_issued[i] - 1) & 1, p.err);
    }
    __syncwarp();
  } else if (warp < kMmaWarp + kIssuers) {
    // ---------------------------------------------------------- MMA issuer --
    const int mi = warp - kMmaWarp;  // issues the tiles == mi (mod kIssuers)
    // One thread; descriptors are the base ones plus constant offsets (the
    // start-address field holds address >> 4; no operand ends above 256 KB,
    // so adding to it never carries into the next field).
    if (lane == 0) {
      RowCursor cur;
      cur.init(p.sched, p.end, p.R, c0, c1, p.nb * 64, row0);
      const uint64_t ad0 = sw128_desc(smem_u32(s.a[0]), 16, 1024);
      constexpr uint32_t kATileDesc = sizeof(s.a[0]) >> 4;
      int lt = 0;
      bool new_group = true;
      while (cur.valid() && !*abort) {
        const int slot = cur.gcount & 1;
        if (new_group && !mbar_wait(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) break;
        bool bad = false;
        const uint64_t bd = sw128_desc(smem_u32(s.q[slot]), 16, 1024);
        for (int t = cur.tile_begin(); t < cur.tile_end(); ++t, ++lt) {
          if (lt % kIssuers != mi) continue;
          const int st = lt % kStages;
          const int buf = lt % kAcc;
          const int ub = lt / kAcc;
          // the scale warps have seen the stage land and filled its scale block
          if (!mbar_wait(&s.sready[st], (lt / kStages) & 1, p.err, abort)) { bad = true; break; }
          if (ub > 0 && !mbar_wait(&s.tempty[buf], (ub - 1) & 1, p.err, abort)) { bad = true; break; }
          tc_fence_after();
          const uint64_t ad = ad0 + static_cast<uint64_t>(st * kATileDesc);
          const uint32_t d = s.tmem_base + static_cast<uint32_t>(buf * 64);
          const uint32_t sfa = s.tmem_base + kSfaCol + kSfStride * static_cast<uint32_t>(st);
          const uint32_t sfb = s.tmem_base + kSfbCol;
          // one K group of 32 elements is 32 bytes of footprint (2 in the address field)
          mma_mxf8f6f4_bs(d, ad, bd, make_idesc_bs(kFmtE2M1, 0, 128, 64, 0u, 0u), sfa, sfb, 0u);
          mma_mxf8f6f4_bs(d, ad + 2, bd + 2, make_idesc_bs(kFmtE2M1, 0, 128, 64, 1u, 0u), sfa, sfb, 1u);
          mma_mxf8f6f4_bs(d, ad + 4, bd + 4, make_idesc_bs(kFmtE2M1, 0, 128, 64, 2u, 0u), sfa, sfb, 1u);
          mma_mxf8f6f4_bs(d, ad + 6, bd + 6, make_idesc_bs(kFmtE2M1, 0, 128, 64, 3u, 0u), sfa, sfb, 1u);
          mma_commit(&s.empty[st]);
          mma_commit(&s.tfull[buf]);
        }
        if (bad) break;
        new_group = cur.next();
        if (new_group) mma_commit(&s.qempty[slot]);
      }
    }
    __syncwarp();
  } else if (warp < kFirstEpiWarp) {
    // --------------------------------------------------------- scale warps --
    // Each warp writes the stage's scale block into the TMEM lane quadrant it
    // may access (warp % 4): lane l, columns j = 0..3 take the scale words of
    // rows 32 j + l, so every quadrant holds the whole block.  The stage's
    // scale block is free once its previous tile's MMAs completed, which its
    // producer waited for before refilling the stage.
    const int quad = warp & 3;
    RowCursor cur;
    cur.init(p.sched, p.end, p.R, c0, c1, p.nb * 64, row0);
    int lt = 0;
    while (cur.valid() && !*abort) {
      bool bad = false;
      for (int t = cur.tile_begin(); t < cur.tile_end(); ++t, ++lt) {
        const int st = lt % kStages;
        if (!mbar_wait_warp(&s.full[st], (lt / kStages) & 1, p.err, abort)) { bad = true; break; }
        uint32_t sfw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          sfw[j] = *reinterpret_cast<const uint32_t*>(s.sf[st] + 128 * j + 4 * lane);
        tmem_st4_sync(s.tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + kSfaCol +
                          kSfStride * static_cast<uint32_t>(st),
                      sfw[0], sfw[1], sfw[2], sfw[3]);
        tc_fence_before();  // the scale block -> the MMA issuer
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sready[st]);
      }
      if (bad) break;
      cur.next();
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quad = warp & 3;
    const int grp = (warp - kFirstEpiWarp) >> 2;  // drains the tiles == grp (mod 2)
    const int tr = quad * 32 + lane;  // token row of the tile == TMEM lane
    RowCursor cur;
    cur.init(p.sched, p.end, p.R, c0, c1, p.nb * 64, row0);
    int lt = 0;
    while (cur.valid() && !*abort) {
      const int slot = cur.gcount & 1;
      const int r = cur.row;
      const int endr = min(p.end[r], p.nb * 64);
      bool waited_q = false, bad = false;
      for (int t = cur.tile_begin(); t < cur.tile_end(); ++t, ++lt) {
        if ((lt & 1) != grp) continue;
        if (!waited_q) {
          if (!mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) { bad = true; break; }
          waited_q = true;
        }
        const int buf = lt % kAcc;
        if (!mbar_wait_warp(&s.tfull[buf], (lt / kAcc) & 1, p.err, abort)) { bad = true; break; }
        tc_fence_after();
        const uint32_t taddr = s.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               static_cast<uint32_t>(buf * 64);
        float v[64];
        tmem_ld64_sync(taddr, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.tempty[buf]);
        const float acc = relu_dot64(v, s.wq[slot]);
        const int col = t * kTileCols + tr;
        if (col < endr) {
          const int64_t o = static_cast<int64_t>(r) * p.ld + col;
          if (p.logits_bf16)
            p.logits_bf16[o] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
          else
            p.logits[o] = acc;
        }
      }
      if (bad) break;
      // A group without tiles here still has its Q waited for before the
      // slot's qempty arrival, so the arrival cannot land in the phase of the
      // group that used the slot two groups earlier.
      if (!waited_q && !mbar_wait_warp(&s.qfull[slot], (cur.gcount >> 1) & 1, p.err, abort)) break;
      const int gslot = slot;
      const bool left = cur.next();
      if (left && lane == 0) mbar_arrive(&s.qempty[gslot]);
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(s.tmem_base, kTmemCols);
  }
}

}  // namespace

size_t candidate_schedule_size(int R) {
  return (static_cast<size_t>(R) + 1 + 3) / 4 * 16;
}

cudaError_t launch_candidate_expand(const CandExpandArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  candidate_expand_kernel<<<a.R, 256, 0, stream>>>(a, dev.err_word);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  schedule_scan_kernel<<<1, 1024, 0, stream>>>(static_cast<int32_t*>(a.schedule), a.R);
  return cudaGetLastError();
}

cudaError_t launch_candidate_logits(const CandLogitsArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream, char* msg, size_t msg_len) {
  const int R = a.num_req * a.next_n;
  CUtensorMap tq;
  {
    const uint64_t dims[2] = {128, static_cast<uint64_t>(R) * 64};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {128, 64};
    if (!encode_tensor_map(&tq, 0, 2, const_cast<uint8_t*>(a.q), dims, strides, box, true, msg,
                           msg_len))
      return cudaErrorInvalidValue;
  }
  CUtensorMap tk;
  {
    // keys as [pages][64 tokens][128 e2m1] in the 4-bit "16 values in 8
    // bytes, padded to 16 in shared memory" type; one box = one page, 128B swizzle
    const uint64_t dims[3] = {128, 64, static_cast<uint64_t>(a.num_pages)};
    const uint64_t strides[2] = {64, static_cast<uint64_t>(a.k_page_stride)};
    const uint32_t box[3] = {128, 64, 1};
    if (!encode_tensor_map(&tk, 2, 3, const_cast<uint8_t*>(a.k_fp4), dims, strides, box, true, msg,
                           msg_len))
      return cudaErrorInvalidValue;
  }
  CParams p;
  p.q_scale = a.q_scale;
  p.w = a.w;
  p.k_fp4 = a.k_fp4;
  p.k_page_stride = a.k_page_stride;
  p.k_sf = a.k_sf;
  p.sf_page_stride = a.sf_page_stride;
  p.num_pages = a.num_pages;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.next_n = a.next_n;
  p.R = R;
  p.sparse_indices = a.sparse_indices;
  p.nb = a.nb;
  p.end = a.end;
  p.sched = static_cast<const int32_t*>(a.schedule);
  p.logits = a.logits;
  p.logits_bf16 = a.logits_bf16;
  p.ld = a.ld;
  p.err = dev.err_word;
  // at least 120 KB so that one CTA (holding all 512 TMEM columns) runs per SM
  const size_t smem = sizeof(CSmem) + 1024 > 120 * 1024 ? sizeof(CSmem) + 1024 : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(candidate_logits_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  candidate_logits_kernel<<<dev.sm_count, kThreads, smem, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace dsa
