// Sparse MLA decode, Eq. (2) of "DeepSeek V3.2-Exp support" (llama.cpp issue
// 16331, section "1. Architecture"): attention of each query row's 128 heads
// over only the k selected latents c_s (576 = 512 latent + 64 rope elements;
// the value is the first 512).
//
// Work unit = one CTA per (row, value half vh, split):
//   * Q of the row (128 heads x 576 bf16, 147 KB) is loaded once by TMA into
//     nine 128B-swizzled [128 x 64] K-chunks;
//   * the split's selected tokens are taken 64 at a time; their latents are
//     gathered by 16-byte cp.async into nine [64 tokens x 64] 128B-swizzled
//     chunks that flow through an 8-slot ring (the chunks outside this CTA's
//     value half first, so they free their slots early);
//   * S = Q K^T (M = 128 heads, N = 64 tokens, K = 576) runs on tcgen05
//     kind::f16 into TMEM;
//   * the softmax warpgroup (one thread per head / TMEM lane) masks invalid
//     tokens, keeps a running max (rescaling O in TMEM only when the max grows
//     by more than 2^8), writes P = exp2(S*scale*log2e - m) as bf16 into a
//     swizzled smem tile;
//   * O[128 x 256] += P V_half runs on tcgen05 with V read MN-major straight
//     from the gathered chunks.
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

constexpr int kThreads = 256;  // warp 0 MMA, warps 1-3 gather, warps 4-7 softmax/epilogue
constexpr int kGather = 96;
constexpr int kRing = 8;
constexpr int kTile = 64;
constexpr int kChunks = 9;       // 576 / 64
constexpr int kSOnly = 5;        // chunks used only by S (other half + rope)
constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kHalf = 256;
constexpr int kTargetCtas = 152;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct MParams {
  const uint16_t* kv;
  int64_t kv_page_stride;  // bytes
  int num_pages;
  const int32_t* bt;
  int64_t bt_stride;
  int next_n;
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
  uint8_t q[kChunks][128 * 128];   // 9 x 16 KB, K-major SW128, rows = heads
  uint8_t p[128 * 128];            // P tile [128 heads x 64 tokens] bf16, K-major SW128
  uint8_t ring[kRing][kTile * 128];  // [64 tokens x 64 elems] bf16 SW128
  const uint8_t* tokptr[2][kTile];
  uint64_t q_full;
  uint64_t chunk_full[kRing], chunk_empty[kRing];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, pv_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int chunk_of(int vh, int q) {
  // S-only chunks first: the other half's four 64-wide blocks, then the rope block.
  if (q < 4) return (vh ? 0 : 4) + q;
  if (q == 4) return 8;
  return 4 * vh + (q - 5);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
  const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
  return lo | (hi << 16);
}

__device__ __forceinline__ float bf16_round(float a) {
  return __bfloat162float(__float2bfloat16_rn(a));
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const MParams p) {
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescS = make_idesc(1, 1, 128, kTile, false, false);
  constexpr uint32_t kIdescPV = make_idesc(1, 1, 128, 64, false, true);
  constexpr int kSCol = 0;      // S buffers at columns [0, 128)
  constexpr int kOCol = 128;    // O half at columns [128, 384)
  extern __shared__ uint8_t smem_raw[];
  MSmem& s = *reinterpret_cast<MSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int row = blockIdx.x;
  const int vh = blockIdx.y;
  const int split = blockIdx.z;
  const int req = row / p.next_n;
  const int s0 = split * p.tokens_per_split;
  const int s1 = min(p.k, s0 + p.tokens_per_split);
  const int ntile = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;
  const int32_t* idx_row = p.idx + static_cast<int64_t>(row) * p.k;

  if (tid == 0) {
    s.abort = 0;
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&s.chunk_full[i], kGather);
      mbar_init(&s.chunk_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_empty[i], 4);
    }
    mbar_init(&s.p_full, 128);
    mbar_init(&s.pv_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile int* abort = &s.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer --
    if (ntile > 0 && mbar_wait(&s.q_full, 0, p.err, abort)) {
      for (int i = 0; i < ntile && !*abort; ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait(&s.s_empty[buf], ((i >> 1) - 1) & 1, p.err, abort)) break;
        tc_fence_after();
        const uint32_t dS = s.tmem_base + kSCol + buf * kTile;
        bool bad = false;
        for (int qq = 0; qq < kChunks; ++qq) {
          const int g = i * kChunks + qq;
          const int slot = g % kRing;
          if (!mbar_wait(&s.chunk_full[slot], (g / kRing) & 1, p.err, abort)) { bad = true; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = smem_u32(s.q[chunk_of(vh, qq)]);
            const uint32_t b0 = smem_u32(s.ring[slot]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(dS, sw128_desc(a0 + 32 * kk, 16, 1024), sw128_desc(b0 + 32 * kk, 16, 1024),
                      kIdescS, (qq | kk) != 0);
            if (qq < kSOnly) mma_commit(&s.chunk_empty[slot]);
          }
          __syncwarp();
        }
        if (bad) break;
        if (lane == 0) mma_commit(&s.s_full[buf]);
        __syncwarp();
        if (!mbar_wait(&s.p_full, i & 1, p.err, abort)) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t pa = smem_u32(s.p);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int slot = (i * kChunks + kSOnly + j) % kRing;
              const uint32_t vb = smem_u32(s.ring[slot]) + 2048 * kk;
              mma_f16(s.tmem_base + kOCol + 64 * j, sw128_desc(pa + 32 * kk, 16, 1024),
                      sw128_desc(vb, 8192, 1024), kIdescPV, (i > 0 || kk > 0));
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_commit(&s.chunk_empty[(i * kChunks + kSOnly + j) % kRing]);
          mma_commit(&s.pv_done);
        }
        __syncwarp();
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- gather --
    const int gt = tid - 32;  // 0..95
    if (gt == 0 && ntile > 0) {
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(&s.q_full, kChunks * 128 * 128);
      for (int c = 0; c < kChunks; ++c) tma_load_2d(s.q[c], &tm_q, &s.q_full, 64 * c, row * kHeads);
    }
    const uint8_t* kvb = reinterpret_cast<const uint8_t*>(p.kv);
    // Token pointers: idx is read two tiles ahead and the block table one tile
    // ahead, so neither load sits on the path that issues a tile's copies.
    auto load_tok = [&](int i) -> int {
      const int pos = s0 + i * kTile + gt;
      return (gt < kTile && i < ntile && pos < s1) ? idx_row[pos] : -1;
    };
    auto load_page = [&](int tok) -> int {
      if (tok < 0) return -1;
      const int64_t pg_i = tok / 64;
      return pg_i < p.bt_stride ? p.bt[static_cast<int64_t>(req) * p.bt_stride + pg_i] : -1;
    };
    auto make_ptr = [&](int tok, int page) -> const uint8_t* {
      if (tok < 0) return nullptr;
      if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, kErrBadIndex);
        return nullptr;
      }
      return kvb + static_cast<int64_t>(page) * p.kv_page_stride +
             static_cast<int64_t>(tok % 64) * (kDqk * 2);
    };
    int tok_a = load_tok(0);
    int tok_b = load_tok(1);
    if (gt < kTile) s.tokptr[0][gt] = make_ptr(tok_a, load_page(tok_a));
    constexpr int kDepth = 4;  // chunks kept in flight per thread
    int issued = 0;            // chunks issued so far (global chunk counter)
    int signalled = 0;
    bool bad = false;
    // Every gather thread passes exactly one named barrier per tile, even after
    // an abort, so no thread can be left waiting on the barrier.
    for (int i = 0; i < ntile; ++i) {
      const int tb = i & 1;
      named_bar_sync(1, kGather);
      if (bad || *abort) {
        bad = true;
        continue;
      }
      int page_b = -1, tok_c = -1;
      if (gt < kTile && i + 1 < ntile) {
        page_b = load_page(tok_b);
        tok_c = load_tok(i + 2);
      }
      for (int qq = 0; qq < kChunks; ++qq) {
        const int g = i * kChunks + qq;
        const int slot = g % kRing;
        if (g >= kRing && !mbar_wait(&s.chunk_empty[slot], ((g / kRing) - 1) & 1, p.err, abort)) {
          bad = true;
          break;
        }
        const int c = chunk_of(vh, qq);
        uint8_t* dst = s.ring[slot];
        for (int piece = gt; piece < kTile * 8; piece += kGather) {
          const int r = piece >> 3, ch = piece & 7;
          const uint8_t* src = s.tokptr[tb][r];
          uint8_t* d = dst + sw128_offset(r, ch);
          if (src) cp_async_16(d, src + c * 128 + ch * 16);
          else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
        ++issued;
        if (issued - signalled > kDepth) {
          cp_async_wait<kDepth>();
          fence_proxy_async_smem();
          mbar_arrive(&s.chunk_full[signalled % kRing]);
          ++signalled;
        }
      }
      if (gt < kTile && i + 1 < ntile) {
        s.tokptr[tb ^ 1][gt] = make_ptr(tok_b, page_b);
        tok_b = tok_c;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (!bad)
      while (signalled < issued) {
        mbar_arrive(&s.chunk_full[signalled % kRing]);
        ++signalled;
      }
  } else {
    // ------------------------------------------------------ softmax / epilogue --
    const int quad = warp & 3;
    const int h = quad * 32 + lane;  // head == TMEM lane
    const uint32_t lane_base = s.tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool bad = false;
    // validity of a tile's 64 selections: lane j of every warp reads entries j
    // and 32 + j, the two ballots give the tile's mask (read one tile ahead)
    auto load_sel = [&](int i, int off) -> int {
      const int pos = s0 + i * kTile + off + lane;
      return (i < ntile && pos < s1) ? idx_row[pos] : -1;
    };
    int sel_lo = load_sel(0, 0), sel_hi = load_sel(0, 32);
    for (int i = 0; i < ntile; ++i) {
      const unsigned m_lo = __ballot_sync(0xffffffffu, sel_lo >= 0);
      const unsigned m_hi = __ballot_sync(0xffffffffu, sel_hi >= 0);
      sel_lo = load_sel(i + 1, 0);
      sel_hi = load_sel(i + 1, 32);
      const int buf = i & 1;
      if (!mbar_wait(&s.s_full[buf], (i >> 1) & 1, p.err, abort)) { bad = true; break; }
      tc_fence_after();
      float x[kTile];
      tmem_ld64_sync(lane_base + kSCol + buf * kTile, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.s_empty[buf]);
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTile; ++j) {
        const bool ok = ((j < 32 ? (m_lo >> j) : (m_hi >> (j - 32))) & 1u) != 0;
        x[j] = ok ? x[j] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[j]);
      }
      // PV(i-1) must be complete before P is overwritten or O rescaled
      if (i > 0 && !mbar_wait(&s.pv_done, (i - 1) & 1, p.err, abort)) { bad = true; break; }
      tc_fence_after();
      const bool grow = mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY);
      const float m_new = grow ? mt : m_run;
      const bool need_rescale = grow && i > 0 && m_run > -INFINITY;
      const float corr = need_rescale ? exp2f(m_run - m_new) : 1.f;
      if (__any_sync(0xffffffffu, need_rescale)) {
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
      l_run *= corr;
      m_run = m_new;
      // P = exp2(x - m) in bf16, row h of the swizzled P tile
      uint8_t* prow = s.p + h * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          e[j] = m_run == -INFINITY ? 0.f : exp2f(x[8 * ch + j] - m_run);
          l_run += bf16_round(e[j]);
        }
        uint4 v;
        v.x = pack_bf16(e[0], e[1]);
        v.y = pack_bf16(e[2], e[3]);
        v.z = pack_bf16(e[4], e[5]);
        v.w = pack_bf16(e[6], e[7]);
        *reinterpret_cast<uint4*>(prow + ((ch ^ (h & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&s.p_full);
    }
    // ---- epilogue: O half of this CTA ----
    if (!bad && ntile > 0 && mbar_wait(&s.pv_done, (ntile - 1) & 1, p.err, abort)) {
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
  if (warp == 0) {
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
  (void)dev;
  const int R = a.num_req * a.next_n;
  const int ns = choose_nsplit(R, a.k);
  const int tiles = (a.k + kTile - 1) / kTile;
  const int tps = ((tiles + ns - 1) / ns) * kTile;
  CUtensorMap tq;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kDqk), static_cast<uint64_t>(R) * kHeads};
    const uint64_t strides[1] = {kDqk * 2};
    const uint32_t box[2] = {64, 128};
    char msg[128];
    if (!encode_tensor_map(&tq, 1, 2, const_cast<uint16_t*>(a.q), dims, strides, box, true, msg,
                           sizeof(msg)))
      return cudaErrorInvalidValue;
  }
  MParams p;
  p.kv = a.kv;
  p.kv_page_stride = a.kv_page_stride;
  p.num_pages = a.num_pages;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.next_n = a.next_n;
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
  const int R = a_in.num_req * a_in.next_n;
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
