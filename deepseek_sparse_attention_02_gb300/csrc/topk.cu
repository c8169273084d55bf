// Exact per-row top-k (the fine-grained token selection of Eq. (2), "DeepSeek
// V3.2-Exp support", section "1. Architecture").
//
// Each row is owned by one thread-block cluster of kC CTAs; CTA c takes the
// c-th contiguous slice of the row.  Histograms are merged across the cluster
// through distributed shared memory, so the row is read from HBM once and the
// later passes run on shared memory.  Clusters loop over rows (persistent).
//
// Selection is a most-significant-digit radix select (8-bit digits) on the
// 64-bit key  (order-preserving u32 of the f32 score) << 32 | ~column,  which
// is unique per element: the k largest keys are the k best scores with ties
// going to the lower column.  It stops as soon as the bin holding the k-th key
// is taken whole, so the column digits are only visited for real ties.
//
//  * full-row path (shorter rows): the slice's keys are staged in shared
//    memory and the radix select runs over all of them;
//  * cutoff path (long rows; the "sampled filtering" of vLLM's persistent
//    top-k in the RepoJournal digest): a strided sample of the row gives a
//    cutoff tau expected to keep about 2k elements; one streaming pass
//    compacts the survivors (key >= tau) into shared memory; the exact radix
//    select then runs on the survivors only.  If the estimate missed (fewer
//    than k survivors, or more than fit) the row is redone by the full-row
//    radix reading global memory, so the result is always exact.
#include <cooperative_groups.h>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kC = 8;       // CTAs per row (cluster size, portable)
constexpr int kT = 256;     // threads per CTA
constexpr int kCap = 8192;  // u32 slots per CTA: staged keys, or survivor (key, column) pairs
constexpr int kPairCap = kCap / 2;
constexpr int kSample = 256;  // sample elements per CTA (cutoff path)

struct TkParams {
  const float* logits;
  int64_t ld;
  const int32_t* row_len;
  int R;
  int k;
  const int32_t* col_blocks;
  int nb;
  int bs;
  int32_t* out;
  int force_path;
  uint32_t* err;
};

struct TkSmem {
  uint32_t data[kCap];
  uint32_t sample[kSample];
  uint32_t hist[256];
  uint32_t chist[2][256];  // read by the other CTAs of the cluster
  uint32_t counter;        // rank 0's is the cluster-wide output cursor
  uint32_t cnt;            // survivors of this CTA (cluster-visible)
  uint32_t overflow;       // cluster-visible
  uint32_t bin, above, binc;
};

__device__ __forceinline__ uint32_t key_of(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0) u = 0;  // -0.0 ranks with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Radix state: after `depth` digits the selected set is every element whose
// top `depth` digits of (key, ~col) are >= (phi, plo).
struct Sel {
  int depth;
  uint32_t phi, plo;
};

__device__ __forceinline__ bool matches(const Sel& s, uint32_t key, uint32_t nidx) {
  const int d = s.depth;
  if (d == 0) return true;
  if (d < 4) return (key >> (32 - 8 * d)) == s.phi;
  if (key != s.phi) return false;
  if (d == 4) return true;
  return (nidx >> (32 - 8 * (d - 4))) == s.plo;
}

__device__ __forceinline__ uint32_t digit(int d, uint32_t key, uint32_t nidx) {
  return d < 4 ? (key >> (24 - 8 * d)) & 255u : (nidx >> (24 - 8 * (d - 4))) & 255u;
}

__device__ __forceinline__ bool selected(const Sel& s, uint32_t key, uint32_t nidx) {
  const int d = s.depth;
  if (d < 4) return (key >> (32 - 8 * d)) >= s.phi;
  if (d == 4) return key >= s.phi;
  if (key != s.phi) return key > s.phi;
  return (nidx >> (32 - 8 * (d - 4))) >= s.plo;
}

// Warp-aggregated histogram increment (all 32 lanes call it).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool valid) {
  const unsigned act = __ballot_sync(0xffffffffu, valid);
  if (valid) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1))
      atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
  }
}

// Element sources.  visit(f) calls f(key, ~col, valid) with every lane of
// every warp taking part in each call (valid = false for padding lanes).
struct SrcGlobal {  // the slice [lo, hi) of a row, read from global memory
  const float* row;
  int lo, hi;
  template <class F>
  __device__ void visit(F&& f) const {
    const int n = hi - lo;
    const int n4 = (n + 3) >> 2;
    const int lim = ((n4 + kT - 1) / kT) * kT;
    for (int i4 = threadIdx.x; i4 < lim; i4 += kT) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int e0 = 4 * i4;
      if (e0 + 3 < n) {
        v = *reinterpret_cast<const float4*>(row + lo + e0);
      } else if (e0 < n) {
        v.x = row[lo + e0];
        if (e0 + 1 < n) v.y = row[lo + e0 + 1];
        if (e0 + 2 < n) v.z = row[lo + e0 + 2];
      }
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        f(key_of(vv[j]), ~static_cast<uint32_t>(lo + e0 + j), e0 + j < n);
    }
  }
};

struct SrcStaged {  // keys of the slice staged in shared memory, in column order
  const uint32_t* keys;
  int lo, n;
  template <class F>
  __device__ void visit(F&& f) const {
    const int n4 = (n + 3) >> 2;
    const int lim = ((n4 + kT - 1) / kT) * kT;
    for (int i4 = threadIdx.x; i4 < lim; i4 += kT) {
      const int e0 = 4 * i4;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (e0 < n) v = *reinterpret_cast<const uint4*>(keys + e0);
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) f(vv[j], ~static_cast<uint32_t>(lo + e0 + j), e0 + j < n);
    }
  }
};

struct SrcPairs {  // survivors: keys[i] at column cols[i]
  const uint32_t* keys;
  const uint32_t* cols;
  int n;
  template <class F>
  __device__ void visit(F&& f) const {
    const int lim = ((n + kT - 1) / kT) * kT;
    for (int i = threadIdx.x; i < lim; i += kT) {
      const bool ok = i < n;
      f(ok ? keys[i] : 0u, ok ? ~cols[i] : 0u, ok);
    }
  }
};

struct SrcKeys {  // a key-only list (the sample)
  const uint32_t* keys;
  int n;
  template <class F>
  __device__ void visit(F&& f) const {
    const int lim = ((n + kT - 1) / kT) * kT;
    for (int i = threadIdx.x; i < lim; i += kT) {
      const bool ok = i < n;
      f(ok ? keys[i] : 0u, 0u, ok);
    }
  }
};

// Cluster-wide radix select: returns the state whose selected set has exactly
// `need` elements over the union of the CTAs' sources (for key-only sources
// with ties at the last digit: the smallest key with at least `need` elements
// at or above it).  `phase` counts passes for the double-buffered cluster
// histograms and advances identically in every CTA of the cluster.
template <class Src>
__device__ Sel cluster_select(const Src& src, uint32_t need, int max_depth, TkSmem& s,
                              cg::cluster_group& cluster, int& phase) {
  Sel st{0, 0u, 0u};
  const int tid = threadIdx.x;
  while (st.depth < max_depth) {
    if (tid < 256) s.hist[tid] = 0;
    __syncthreads();
    const int d = st.depth;
    src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
      const bool m = valid && matches(st, key, nidx);
      hist_add(s.hist, digit(d, key, nidx), m);
    });
    __syncthreads();
    const int buf = phase & 1;
    ++phase;
    if (tid < 256) s.chist[buf][tid] = s.hist[tid];
    cluster.sync();
    if (tid < 256) {
      uint32_t tot = 0;
#pragma unroll
      for (int r = 0; r < kC; ++r) tot += cluster.map_shared_rank(&s.chist[buf][0], r)[tid];
      s.hist[tid] = tot;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      const int lane = tid;
      uint32_t h[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = s.hist[255 - 8 * lane - j];
        sum += h[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      uint32_t above = incl - sum;
      if (above < need && need <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + h[j] >= need) {
            s.bin = 255 - 8 * lane - j;
            s.above = above;
            s.binc = h[j];
            break;
          }
          above += h[j];
        }
      }
    }
    __syncthreads();
    const uint32_t b = s.bin;
    need -= s.above;
    if (d < 4) st.phi = (st.phi << 8) | b;
    else st.plo = (st.plo << 8) | b;
    st.depth = d + 1;
    const bool done = s.binc == need;
    __syncthreads();
    if (done) break;
  }
  return st;
}

__device__ __forceinline__ int32_t map_col(const TkParams& p, int row, uint32_t col) {
  if (!p.col_blocks) return static_cast<int32_t>(col);
  if (col / static_cast<uint32_t>(p.bs) >= static_cast<uint32_t>(p.nb)) {
    raise_error(p.err, kErrBadIndex);
    return -1;
  }
  const int64_t blk = p.col_blocks[static_cast<int64_t>(row) * p.nb + col / p.bs];
  return static_cast<int32_t>(blk * p.bs + col % p.bs);
}

// Writes every selected element of the source to out[row], in any order.
template <class Src>
__device__ void emit(const Src& src, const Sel& st, const TkParams& p, int row, TkSmem& s,
                     cg::cluster_group& cluster) {
  uint32_t* cursor = cluster.map_shared_rank(&s.counter, 0);
  int32_t* out = p.out + static_cast<int64_t>(row) * p.k;
  const int lane = threadIdx.x & 31;
  src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
    const bool take = valid && selected(st, key, nidx);
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (m == 0) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(cursor, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (take) {
      const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
      if (pos < static_cast<uint32_t>(p.k)) out[pos] = map_col(p, row, ~nidx);
    }
  });
}

__global__ void __launch_bounds__(kT, 4) topk_kernel(const TkParams p) {
  extern __shared__ uint8_t smem_raw[];
  TkSmem& s =
      *reinterpret_cast<TkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int cid = blockIdx.x / kC;
  const int ncl = gridDim.x / kC;
  const int tid = threadIdx.x;
  int phase = 0;

  for (int row = cid; row < p.R; row += ncl) {
    const float* rowp = p.logits + static_cast<int64_t>(row) * p.ld;
    int L = p.row_len[row];
    if (L < 0) L = 0;
    if (L > p.ld) {
      if (tid == 0 && rank == 0) raise_error(p.err, kErrBadIndex);
      L = static_cast<int>(p.ld);
    }
    const int S = (((L + kC - 1) / kC) + 3) & ~3;
    const int lo = min(L, rank * S);
    const int hi = min(L, lo + S);
    int32_t* out = p.out + static_cast<int64_t>(row) * p.k;

    if (L <= p.k) {
      // every column is selected; the tail is -1 (no cluster communication)
      for (int c = lo + tid; c < hi; c += kT) out[c] = map_col(p, row, c);
      const int pad = p.k - L;
      const int per = (pad + kC - 1) / kC;
      const int a = L + rank * per, b = min(p.k, a + per);
      for (int c = a + tid; c < b; c += kT) out[c] = -1;
      continue;
    }

    if (tid == 0) {
      s.counter = 0;
      s.overflow = 0;
      s.cnt = 0;
    }
    const bool cutoff =
        p.force_path == 2 || (p.force_path == 0 && L >= (p.k < 1024 ? 98304 : 65536));
    cluster.sync();  // counters reset everywhere before anyone emits

    bool done = false;
    if (cutoff) {
      // 1. sample -> cutoff tau expected to keep about 2k elements
      const int n = hi - lo;
      const int ns = min(kSample, n);
      const int stride = ns > 0 ? n / ns : 1;
      for (int i = tid; i < ns; i += kT) s.sample[i] = key_of(rowp[lo + i * stride]);
      __syncthreads();
      int NS = 0;
      for (int r = 0; r < kC; ++r) {
        const int lr = min(L, r * S), hr = min(L, lr + S);
        NS += min(kSample, hr - lr);
      }
      const double want = 2.0 * p.k * static_cast<double>(NS) / static_cast<double>(L);
      const uint32_t q = static_cast<uint32_t>(fmin(static_cast<double>(NS), ceil(want)));
      SrcKeys sk{s.sample, ns};
      // two digits (sign, exponent, 7 mantissa bits) place tau within ~1 % of
      // the sample's q-th key, which is all the estimate needs
      const Sel ts = cluster_select(sk, q > 0 ? q : 1u, 2, s, cluster, phase);
      const uint32_t tau = ts.phi << (32 - 8 * ts.depth);
      // 2. one streaming pass: compact the survivors (key >= tau)
      uint32_t* skeys = s.data;
      uint32_t* scols = s.data + kPairCap;
      SrcGlobal g{rowp, lo, hi};
      const int lane = tid & 31;
      g.visit([&](uint32_t key, uint32_t nidx, bool valid) {
        const bool keep = valid && key >= tau;
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (m == 0) return;
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&s.cnt, static_cast<uint32_t>(__popc(m)));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (keep) {
          const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
          if (pos < kPairCap) {
            skeys[pos] = key;
            scols[pos] = ~nidx;
          }
        }
      });
      __syncthreads();
      if (tid == 0 && s.cnt > kPairCap) s.overflow = 1;
      cluster.sync();
      uint32_t total = 0, over = 0;
      for (int r = 0; r < kC; ++r) {
        total += *cluster.map_shared_rank(&s.cnt, r);
        over |= *cluster.map_shared_rank(&s.overflow, r);
      }
      if (!over && total >= static_cast<uint32_t>(p.k)) {
        SrcPairs sp{skeys, scols, static_cast<int>(min(s.cnt, static_cast<uint32_t>(kPairCap)))};
        const Sel st = cluster_select(sp, p.k, 8, s, cluster, phase);
        emit(sp, st, p, row, s, cluster);
        done = true;
      } else if (tid == 0 && rank == 0) {
        raise_error(p.err, kErrCapacity);
      }
    }
    if (!done) {
      const int n = hi - lo;
      // full-row radix select (also the exact redo of a missed cutoff)
      if (!cutoff && n <= kCap) {
        for (int i4 = tid; 4 * i4 < n; i4 += kT) {
          const int e0 = 4 * i4;
          if (e0 + 3 < n) {
            const float4 v = *reinterpret_cast<const float4*>(rowp + lo + e0);
            *reinterpret_cast<uint4*>(s.data + e0) =
                make_uint4(key_of(v.x), key_of(v.y), key_of(v.z), key_of(v.w));
          } else {
            for (int j = e0; j < n; ++j) s.data[j] = key_of(rowp[lo + j]);
          }
        }
        __syncthreads();
        SrcStaged ss{s.data, lo, n};
        const Sel st = cluster_select(ss, p.k, 8, s, cluster, phase);
        emit(ss, st, p, row, s, cluster);
      } else {
        SrcGlobal g{rowp, lo, hi};
        const Sel st = cluster_select(g, p.k, 8, s, cluster, phase);
        emit(g, st, p, row, s, cluster);
      }
    }
    cluster.sync();  // all emits done before the counters are reused
  }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const size_t smem = sizeof(TkSmem) + 16;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  TkParams p{a.logits, a.ld,  a.row_len, a.R,          a.k,          a.col_blocks,
             a.nb,     a.block_size, a.out, a.force_path, dev.err_word};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  cfg.gridDim = dim3(kC * 64);
  e = cudaOccupancyMaxActiveClusters(&max_clusters, topk_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) max_clusters = 1;
  const int ncl = a.R < max_clusters ? a.R : max_clusters;
  cfg.gridDim = dim3(kC * ncl);
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace dsa
