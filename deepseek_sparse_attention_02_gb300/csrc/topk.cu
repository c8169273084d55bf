// Exact per-row top-k (the fine-grained token selection of Eq. (2), "DeepSeek
// V3.2-Exp support", section "1. Architecture").
//
// One CTA of 1024 threads owns a row (persistent over rows, one CTA per SM).
// Every radix pass synchronises with __syncthreads only: measured on GB300,
// the cross-CTA histogram merges of a cluster-per-row design cost ~2-3 us per
// pass.  When the rows are few (at most half the SM count) a second CTA per
// row (a cluster of two) takes half of the one streaming pass below: that pass
// is bound by the loads one CTA keeps in flight (~26 B/clk from L2), not by
// its instructions, so two SMs halve it; the select itself stays on one CTA.
//
// Selection is a most-significant-digit radix select (11-bit digits) on the
// 64-bit key  (order-preserving u32 of the f32 score) << 32 | ~column,  which
// is unique per element: the k largest keys are the k best scores with ties
// going to the lower column.  It stops as soon as the bin holding the k-th key
// is taken whole, so the column digits are only visited for real ties.
//
//  * staged path (rows shorter than 8k, up to kStage scores): the row's keys
//    are staged in shared memory and the radix select runs over all of them;
//  * cutoff path (longer rows; the "sampled filtering" of vLLM's persistent
//    top-k in the RepoJournal digest): the row's score histogram, when the
//    indexer built one (12-bit order-key prefix, every logit counted), gives
//    the exact cutoff at once: tau = the lower edge of the bin holding the
//    k-th largest score, which keeps k + (that bin's count) at most;
//    otherwise a sample of the row (runs of 8 scores spread over it) gives a
//    cutoff tau expected to keep about 2k elements;
//    one streaming pass compacts the survivors (key >= tau) into shared
//    memory; the exact select then runs on the survivors only (its first
//    digit linear in the key over [tau, largest survivor]).  If the
//    estimate missed (fewer than k survivors, or more than fit) the row is
//    redone by the radix select reading the row from global memory, so the
//    result is always exact.
#include <cooperative_groups.h>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kT = 1024;                // threads per CTA
constexpr int kWarps = kT / 32;
constexpr int kStage = 40960;           // u32 slots: staged keys, or survivor pairs
constexpr int kWarpCap = kStage / 2 / kWarps;  // survivor pairs per warp (640)
// Cutoff-path sample: kGroups runs of 8 consecutive scores spread evenly over
// the row (one 32-byte sector each).
constexpr int kGroups = 256;
constexpr int kSample = 8 * kGroups;
static_assert(kSample / 4 <= kT, "the sample is loaded as one float4 per thread");

struct TkParams {
  const void* logits;  // f32 or bf16 [R, ld]
  int64_t ld;
  const int32_t* row_len;
  int R;
  int k;
  const int32_t* col_blocks;
  int nb;
  int bs;
  int32_t* out;
  int force_path;
  uint32_t* hist;  // null, or [R, kHistBins] score histograms; every row's is cleared
  uint32_t* err;
};

struct TkSmem {
  uint32_t data[kStage];  // staged keys | survivor keys (warp regions) + columns
  uint32_t sample[kSample];
  uint32_t tau_bins[4096];  // the cutoff estimate's histogram (its own: the second CTA of a
                            // pair may already be writing survivors into rank 0's data)
  uint32_t hist[2048];    // radix histogram (kBins)
  uint32_t wscan[kWarps]; // per-warp scan totals
  uint32_t wsum[2 * kWarps];  // per-region survivor counts (a region per warp of the row's CTAs)
  uint32_t wmax[2 * kWarps];  // per-region largest survivor key
  uint32_t counter;       // output cursor
  uint32_t bin, above, binc;
  uint32_t ncand;         // candidates gathered from the boundary bin
  uint32_t stotal, smax, sover;  // survivors, their largest key, a region overflowed
  uint64_t thr;           // the select's result
};

__device__ __forceinline__ uint32_t key_of(float x) { return order_key(x); }

// Radix state: the selected set is every element whose top kb bits of key and
// (once kb == 32) top ib bits of ~column are >= (phi, plo).  Digits are up to
// kDigit bits wide; key digits may start at any bit (the survivor select
// starts at the highest bit where the survivors differ).
constexpr int kDigit = 11;
constexpr int kBins = 1 << kDigit;
struct Sel {
  int kb, ib;
  uint32_t phi, plo;
};

__device__ __forceinline__ bool matches(const Sel& s, uint32_t key, uint32_t nidx) {
  if (s.kb < 32) return s.kb == 0 || (key >> (32 - s.kb)) == s.phi;
  if (key != s.phi) return false;
  return s.ib == 0 || (nidx >> (32 - s.ib)) == s.plo;
}

// Width of the next digit, and the digit itself.
__device__ __forceinline__ int digit_bits(const Sel& s) {
  return min(kDigit, 32 - (s.kb < 32 ? s.kb : s.ib));
}
__device__ __forceinline__ uint32_t digit(const Sel& s, int w, uint32_t key, uint32_t nidx) {
  return s.kb < 32 ? (key >> (32 - s.kb - w)) & ((1u << w) - 1u)
                   : (nidx >> (32 - s.ib - w)) & ((1u << w) - 1u);
}

// The smallest 64-bit (key, ~column) value whose leading fixed bits equal the
// state's prefix: once the select is done, the selected set is exactly the
// elements whose (key << 32 | ~column) is >= this threshold.
__device__ __forceinline__ uint64_t threshold(const Sel& s) {
  const uint32_t hi = s.kb == 0 ? 0u : (s.kb == 32 ? s.phi : s.phi << (32 - s.kb));
  const uint32_t lo = s.ib == 0 ? 0u : (s.ib == 32 ? s.plo : s.plo << (32 - s.ib));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t pack(uint32_t key, uint32_t nidx) {
  return (static_cast<uint64_t>(key) << 32) | nidx;
}

// Read-only global loads as volatile asm: they are issued in program order, so
// a batch of them is in flight before the first one is consumed.
__device__ __forceinline__ float4 ldg_nc4(const float* ptr) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr));
  return v;
}
__device__ __forceinline__ float ldg_nc(const float* ptr) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
  return v;
}

// A row of scores in global memory: f32, or bf16 widened to f32 on load (an
// exact widening, so a bf16 row selects as the f32 row of the same values).
// load4 needs e0 % 4 == 0 (16- or 8-byte aligned loads).
template <class T>
struct RowPtr;
template <>
struct RowPtr<float> {
  const float* p;
  __device__ float4 load4(int64_t e0) const { return ldg_nc4(p + e0); }
  __device__ float load1(int64_t e) const { return ldg_nc(p + e); }
  __device__ RowPtr offset(int64_t c) const { return {p + c}; }
};
template <>
struct RowPtr<uint16_t> {
  const uint16_t* p;
  __device__ float4 load4(int64_t e0) const {
    uint32_t a, b;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "l"(p + e0));
    return make_float4(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u),
                       __uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
  }
  __device__ float load1(int64_t e) const {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p + e));
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  __device__ RowPtr offset(int64_t c) const { return {p + c}; }
};

// Element sources.  visit(f) calls f(key, ~col, valid) with every lane of a
// warp taking part in each call (valid = false for padding lanes).

template <class T>
struct SrcGlobal {  // the row [0, n), read from global memory
  RowPtr<T> row;
  int n;
  static constexpr int kB = 4;  // float4 loads in flight per thread
  __device__ float4 load4(int e0) const {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e0 + 3 < n) {
      v = row.load4(e0);
    } else if (e0 < n) {
      v.x = row.load1(e0);
      if (e0 + 1 < n) v.y = row.load1(e0 + 1);
      if (e0 + 2 < n) v.z = row.load1(e0 + 2);
    }
    return v;
  }
  template <class F>
  __device__ void visit(F&& f) const {
    const int n4 = (n + 3) >> 2;
    for (int base = 0; base < n4; base += kB * kT) {  // same trip count in every thread
      float4 v[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) v[b] = load4(4 * (base + b * kT + threadIdx.x));
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int e0 = 4 * (base + b * kT + threadIdx.x);
        const float vv[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) f(key_of(vv[j]), ~static_cast<uint32_t>(e0 + j), e0 + j < n);
      }
    }
  }
};

struct SrcStaged {  // the row's keys staged in shared memory, in column order
  const uint32_t* keys;
  int n;
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
      for (int j = 0; j < 4; ++j) f(vv[j], ~static_cast<uint32_t>(e0 + j), e0 + j < n);
    }
  }
};

// Survivors: warp w's region is keys/cols [w*kWarpCap, (w+1)*kWarpCap); the
// row's first CTA filled cnt[w] slots from the bottom, a second CTA (if any)
// cnt[kWarps + w] slots from the top (cnt[w] + cnt[kWarps + w] <= kWarpCap,
// else the row overflowed and is not visited this way).
struct SrcPairs {
  const uint32_t* keys;
  const uint32_t* cols;
  const uint32_t* cnt;
  template <class F>
  __device__ void visit(F&& f) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w0 = warp * kWarpCap;  // each warp walks its own region
    const int n0 = static_cast<int>(cnt[warp]);
    const int n = n0 + static_cast<int>(cnt[kWarps + warp]);
    const int lim = (n + 31) & ~31;
    for (int i = lane; i < lim; i += 32) {
      const bool ok = i < n;
      const int j = w0 + (i < n0 ? i : kWarpCap - 1 - (i - n0));
      f(ok ? keys[j] : 0u, ok ? ~cols[j] : 0u, ok);
    }
  }
};

// One histogram pass: bin(key, ~col) gives each element's bin in [0, kBins)
// or -1 for elements outside the current selection.  Leaves in s.bin the bin
// holding the need-th largest element (counting bins from the top), in
// s.above the elements of the higher bins and in s.binc the bin's own count.
// Histogram increments are plain shared-memory atomics: measured on GB300
// over 2048 normal scores, a 256-bin pass costs ~0.6-0.9 k cycles this way
// against 3-13 k cycles when equal bins are first combined with
// __match_any_sync.
template <class Src, class Bin>
__device__ void hist_pass(const Src& src, const Bin& bin, uint32_t need, TkSmem& s) {
  constexpr int kPer = kBins / kT;  // bins per thread in the scan
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kBins; i += kT) s.hist[i] = 0;
  __syncthreads();
  src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
    const int b = valid ? bin(key, nidx) : -1;
    if (b >= 0) atomicAdd(&s.hist[b], 1u);
  });
  __syncthreads();
  // thread t owns bins [kBins - kPer*(t+1), kBins - kPer*t), walked downwards
  const int top = kBins - kPer * tid - 1;
  uint32_t h[kPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    h[j] = s.hist[top - j];
    sum += h[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s.wscan[warp] = incl;
  __syncthreads();
  const uint32_t wt = s.wscan[lane];
  uint32_t wincl = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += v;
  }
  uint32_t above = __shfl_sync(0xffffffffu, wincl - wt, warp) + incl - sum;
  if (above < need && need <= above + sum) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (above + h[j] >= need) {
        s.bin = static_cast<uint32_t>(top - j);
        s.above = above;
        s.binc = h[j];
        break;
      }
      above += h[j];
    }
  }
  if (tid == 0) s.ncand = 0;
  __syncthreads();
}

constexpr uint32_t kCandCap = 512;  // boundary-bin elements ranked directly
static_assert(2 * kCandCap <= kSample, "the candidate list aliases the sample");

// Gathers the n elements with in_bin(key, ~col) (n <= kCandCap) and returns the
// (key, ~col) value of the need-th largest of them (keys are unique, so
// exactly one has rank need - 1).
template <class Src, class In>
__device__ uint64_t rank_finish(const Src& src, const In& in_bin, uint32_t n, uint32_t need,
                                TkSmem& s) {
  uint64_t* cand = reinterpret_cast<uint64_t*>(s.sample);  // free once tau is known
  src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
    if (valid && in_bin(key, nidx)) cand[atomicAdd(&s.ncand, 1u)] = pack(key, nidx);
  });
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n; i += kT) {
    const uint64_t c = cand[i];
    uint32_t r = 0;
    for (uint32_t j = 0; j < n; ++j) r += cand[j] > c ? 1u : 0u;
    if (r == need - 1) s.thr = c;
  }
  __syncthreads();
  const uint64_t thr = s.thr;
  __syncthreads();
  return thr;
}

// Radix select from the state `st`: returns the threshold whose selected set
// (elements with (key << 32 | ~col) >= it) has exactly `need` elements over
// the source.  Digits are taken from the top; once the bin holding the
// need-th element has few enough elements they are ranked directly.
template <class Src>
__device__ uint64_t radix_select(const Src& src, uint32_t need, Sel st, TkSmem& s) {
  for (;;) {
    const int w = digit_bits(st);
    hist_pass(src, [&](uint32_t key, uint32_t nidx) {
      return matches(st, key, nidx) ? static_cast<int>(digit(st, w, key, nidx)) : -1;
    }, need, s);
    const uint32_t b = s.bin, binc = s.binc;
    need -= s.above;
    if (st.kb < 32) {
      st.phi = st.kb == 0 ? b : (st.phi << w) | b;
      st.kb += w;
    } else {
      st.plo = st.ib == 0 ? b : (st.plo << w) | b;
      st.ib += w;
    }
    if (binc == need) return threshold(st);  // the boundary bin is taken whole
    if (binc <= kCandCap)
      return rank_finish(src, [&](uint32_t key, uint32_t nidx) { return matches(st, key, nidx); },
                         binc, need, s);
    __syncthreads();
  }
}

// Cutoff estimate: the lower edge of the 12-bit key prefix (sign, exponent,
// 3 mantissa bits) bin that holds the q-th largest of the sample keys, from
// their 4096-bin histogram in `bins` (shared memory) and a block scan from the
// top bin down.  Keeping every key >= that edge keeps at least q / n of the
// row (n keys sampled) in expectation.
__device__ uint32_t tau_from_bins(uint32_t q, const uint32_t* bins, TkSmem& s) {
  constexpr int kTauBins = 4096, kPer = kTauBins / kT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // thread t owns bins [kTauBins - kPer*(t+1), kTauBins - kPer*t), walked downwards
  const int top = kTauBins - kPer * tid - 1;
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) sum += bins[top - j];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s.wscan[warp] = incl;
  __syncthreads();
  const uint32_t wt = s.wscan[lane];
  uint32_t wincl = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += v;
  }
  uint32_t above = __shfl_sync(0xffffffffu, wincl - wt, warp) + incl - sum;
  if (above < q && q <= above + sum) {
    for (int j = 0; j < kPer; ++j) {
      above += bins[top - j];
      if (above >= q) {
        s.bin = static_cast<uint32_t>(top - j);
        break;
      }
    }
  }
  __syncthreads();
  const uint32_t tau = s.bin << 20;
  __syncthreads();
  return tau;
}

// Cutoff from the row's score histogram h (kHistBins counts of the 12-bit
// key prefix, bin b = keys [b << kHistShift, (b + 1) << kHistShift)): the
// lower edge of the bin holding the k-th largest score, so that every score
// of the higher bins (fewer than k) and the whole boundary bin survive.
// Thread t scans bins [kHistBins - 4(t+1), kHistBins - 4t) downwards.  Returns
// false when the histogram does not count exactly L scores (it was not built
// for this row): the caller then estimates the cutoff from a sample.
__device__ bool hist_tau(const uint32_t* h, int L, uint32_t k, TkSmem& s, uint32_t* tau) {
  constexpr int kPer = kHistBins / kT;
  static_assert(kPer == 4, "one 16-byte load of bins per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int top = kHistBins - kPer * tid - 1;
  // plain (coherent) load: this kernel clears the histogram after reading it
  const uint4 v = *reinterpret_cast<const uint4*>(h + top - 3);
  const uint32_t hh[4] = {v.w, v.z, v.y, v.x};  // bins top, top-1, top-2, top-3
  const uint32_t sum = (hh[0] + hh[1]) + (hh[2] + hh[3]);
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s.wscan[warp] = incl;
  __syncthreads();
  const uint32_t wt = s.wscan[lane];
  uint32_t wincl = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += t;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, wincl, 31);
  uint32_t above = __shfl_sync(0xffffffffu, wincl - wt, warp) + incl - sum;
  if (above < k && k <= above + sum) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (above + hh[j] >= k) {
        s.bin = static_cast<uint32_t>(top - j);
        break;
      }
      above += hh[j];
    }
  }
  __syncthreads();
  *tau = s.bin << kHistShift;
  __syncthreads();
  return total == static_cast<uint32_t>(L);
}

// Clears a row's histogram (all threads of one CTA).
__device__ __forceinline__ void clear_hist(uint32_t* h) {
  static_assert(kHistBins == 4 * kT, "one 16-byte store per thread");
  reinterpret_cast<uint4*>(h)[threadIdx.x] = make_uint4(0, 0, 0, 0);
}

// One streaming pass over the columns [col0, col0 + g.n) of the row (g.row
// points at column col0): every element with key >= tau goes to its warp's
// region of (keys, cols), [w*kWarpCap, (w+1)*kWarpCap), filled from the bottom
// (top = false) or from the top; the warp keeps its running count in a
// register, so the pass takes no atomics.  wsum[w] receives the warp's count
// (the caller treats the row as overflowed if the counts of a region exceed
// kWarpCap; slots past kWarpCap are not written) and wmax[w] its largest kept
// key (0 if none).  The destinations may be another CTA's shared memory
// (generic addresses in the cluster window).  For tau above key(+0.0),
// key_of(x) >= tau is exactly the signed compare of x's bits with tau's float
// bits (negative values, -0.0 and -NaN fall below, +NaN above, as in key_of):
// one instruction per element.
template <bool kPositiveTau, bool kTop, class T>
__device__ void compact(const SrcGlobal<T>& g, uint32_t col0, uint32_t tau, uint32_t* keys,
                        uint32_t* cols, uint32_t* wsum, uint32_t* wmax) {
  constexpr int kB = 4;  // float4 loads per batch
  const int n = g.n;
  const int n4 = (n + 3) >> 2;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint32_t* wkeys = keys + warp * kWarpCap;
  uint32_t* wcols = cols + warp * kWarpCap;
  const int32_t tbits = static_cast<int32_t>(tau & 0x7fffffffu);
  uint32_t kmax = 0, wcount = 0;
  for (int base = 0; base < n4; base += kB * kT) {
    float4 v[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) v[b] = g.load4(4 * (base + b * kT + threadIdx.x));
    uint32_t mask = 0;  // bit 4b + j: element j of load b is kept
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const float vv[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool keep = kPositiveTau ? static_cast<int32_t>(__float_as_uint(vv[j])) >= tbits
                                       : key_of(vv[j]) >= tau;
        mask |= (keep ? 1u : 0u) << (4 * b + j);
      }
    }
    if (4 * (base + kB * kT) > n) {  // the last batch: drop the elements past the row
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int e0 = 4 * (base + b * kT + threadIdx.x);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j >= n) mask &= ~(1u << (4 * b + j));
      }
    }
    const uint32_t c = __popc(mask);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    // survivors are few: walk the set bits, re-reading each kept score (an L1
    // hit) rather than selecting it from the registers by a dynamic index
    uint32_t pos = wcount + incl - c;
    while (mask != 0) {
      const int bit = __ffs(mask) - 1;
      mask &= mask - 1;
      const int e = 4 * (base + (bit >> 2) * kT + threadIdx.x) + (bit & 3);
      const uint32_t key = key_of(g.row.load1(e));
      kmax = max(kmax, key);
      if (pos < static_cast<uint32_t>(kWarpCap)) {
        const uint32_t j = kTop ? kWarpCap - 1 - pos : pos;
        wkeys[j] = key;
        wcols[j] = col0 + static_cast<uint32_t>(e);
      }
      ++pos;
    }
    wcount += wtot;
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    wsum[warp] = wcount;
    wmax[warp] = kmax;
  }
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
__device__ void emit(const Src& src, uint64_t thr, const TkParams& p, int row, TkSmem& s) {
  int32_t* out = p.out + static_cast<int64_t>(row) * p.k;
  const int lane = threadIdx.x & 31;
  src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
    const bool take = valid && pack(key, nidx) >= thr;
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (m == 0) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&s.counter, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (take) {
      const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
      if (pos < static_cast<uint32_t>(p.k)) out[pos] = map_col(p, row, ~nidx);
    }
  });
}

// Select and output over the survivors of the cutoff path, whose keys all
// lie in [tau, kmax]: the first digit is linear in the key, (key - tau) >>
// shift over kBins bins, so the survivors spread evenly over the bins even
// when their range crosses an exponent boundary (where a leading-bits digit
// would put most of them in one bin).  One more pass then writes the elements
// of the bins above the boundary bin and collects the boundary bin's (at most
// kCandCap), which are ranked and the top ones written (one pass fewer than a
// select that gathers the boundary bin, then an output pass: 23.3 -> 22.1 us
// at 64 x 131072).  Heavy ties fall back to the leading-bits radix and emit.
template <class Src>
__device__ void survivor_select_emit(const Src& src, uint32_t need, uint32_t tau, uint32_t kmax,
                                     const TkParams& p, int row, TkSmem& s) {
  const uint32_t span = kmax - tau;
  const int shift = span < static_cast<uint32_t>(kBins) ? 0 : 32 - kDigit - __clz(span);
  hist_pass(src, [&](uint32_t key, uint32_t) {
    return key >= tau ? static_cast<int>((key - tau) >> shift) : -1;
  }, need, s);
  const uint32_t b = s.bin, binc = s.binc;
  const uint32_t rest = need - s.above;
  if (binc <= kCandCap) {
    int32_t* out = p.out + static_cast<int64_t>(row) * p.k;
    const int lane = threadIdx.x & 31;
    uint64_t* cand = reinterpret_cast<uint64_t*>(s.sample);  // free once tau is known
    src.visit([&](uint32_t key, uint32_t nidx, bool valid) {
      const int bb = (valid && key >= tau) ? static_cast<int>((key - tau) >> shift) : -1;
      if (bb == static_cast<int>(b)) cand[atomicAdd(&s.ncand, 1u)] = pack(key, nidx);
      const bool take = bb > static_cast<int>(b);
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (m == 0) return;
      uint32_t base = 0;
      if (lane == 0) base = atomicAdd(&s.counter, static_cast<uint32_t>(__popc(m)));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (take) {
        const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < static_cast<uint32_t>(p.k)) out[pos] = map_col(p, row, ~nidx);
      }
    });
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < binc; i += kT) {
      const uint64_t c = cand[i];
      uint32_t r = 0;
      for (uint32_t q = 0; q < binc; ++q) r += cand[q] > c ? 1u : 0u;
      if (r < rest) {
        const uint32_t pos = atomicAdd(&s.counter, 1u);
        if (pos < static_cast<uint32_t>(p.k)) out[pos] = map_col(p, row, ~static_cast<uint32_t>(c));
      }
    }
    return;
  }
  __syncthreads();
  const uint32_t x = tau ^ kmax;
  const int nb = x == 0 ? 32 : __clz(x);
  const Sel st0{nb, 0, nb == 0 ? 0u : (nb == 32 ? kmax : kmax >> (32 - nb)), 0u};
  const uint64_t thr = radix_select(src, need, st0, s);
  emit(src, thr, p, row, s);
}

// kCsize = CTAs per row: 1, or 2 (a cluster).  The two are separate kernels:
// measured on GB300, merely containing cluster instructions cost the one-CTA
// kernel ~2 us per launch.
template <int kCsize, class T>
__global__ void __launch_bounds__(kT, 1) topk_kernel(const TkParams p) {
  extern __shared__ uint8_t smem_raw[];
  TkSmem& s =
      *reinterpret_cast<TkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  pdl_launch_dependents_and_wait();
  // With two CTAs per row (a cluster of two, used when the rows are few) both
  // derive the same cutoff from the row's sample, each compacts half of the
  // row, rank 1 into regions kWarps..2 kWarps-1 of rank 0's shared memory, and
  // rank 0 runs the exact select and the output.
  constexpr int csize = kCsize;
  int rank = 0;
  if constexpr (kCsize > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
  TkSmem* s0p = &s;
  if constexpr (kCsize > 1) s0p = cg::this_cluster().map_shared_rank(&s, 0);
  TkSmem& s0 = *s0p;

  for (int row = blockIdx.x / csize; row < p.R; row += gridDim.x / csize) {
    const RowPtr<T> rowp{static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ld};
    int L = p.row_len[row];
    if (L < 0) L = 0;
    if (L > p.ld) {
      if (tid == 0) raise_error(p.err, kErrBadIndex);
      L = static_cast<int>(p.ld);
    }
    int32_t* out = p.out + static_cast<int64_t>(row) * p.k;
    uint32_t* const hrow = p.hist ? p.hist + static_cast<int64_t>(row) * kHistBins : nullptr;

    if (L <= p.k) {
      // every column is selected; the tail is -1
      if (rank == 0) {
        for (int c = tid; c < p.k; c += kT) out[c] = c < L ? map_col(p, row, c) : -1;
        if (hrow) clear_hist(hrow);
      }
      continue;
    }

    if (tid == 0) s.counter = 0;
    __syncthreads();
    // the cutoff path keeps ~2k survivors, so it pays once the row is several
    // times k long (measured at 64 x 32768, k = 2048: 16.8 us against 27.5 us
    // staged); rows beyond the staging capacity always take it
    const bool cutoff =
        p.force_path == 2 ||
        (p.force_path == 0 && (L > kStage || static_cast<int64_t>(L) >= 8ll * p.k));
    bool done = false;
    if (cutoff) {
      // 1. the cutoff tau: exact from the row's histogram, or from a sample
      // (expected to keep about 2k elements; rows shorter than the sample are
      // taken whole)
      uint32_t tau = 0;
      const bool exact = hrow && hist_tau(hrow, L, static_cast<uint32_t>(p.k), s, &tau);
      if (!exact) {
        // The sample's keys go straight from the loads into the cutoff
        // histogram (its bins are cleared while the loads are in flight).
        constexpr int kTauBins = 4096;
        const int ns = L >= kSample ? kSample : L;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (L >= kSample && tid < kSample / 4) {
          // float4 tid of the sample: group tid / 2, half tid % 2
          const int64_t g0 =
              ((static_cast<int64_t>(tid >> 1) * (L - 8)) / (kGroups - 1)) & ~3ll;
          v = rowp.load4(g0 + 4 * (tid & 1));
        }
        for (int i = tid; i < kTauBins; i += kT) s.tau_bins[i] = 0;
        __syncthreads();
        if (L >= kSample) {
          if (tid < kSample / 4) {
            atomicAdd(&s.tau_bins[key_of(v.x) >> 20], 1u);
            atomicAdd(&s.tau_bins[key_of(v.y) >> 20], 1u);
            atomicAdd(&s.tau_bins[key_of(v.z) >> 20], 1u);
            atomicAdd(&s.tau_bins[key_of(v.w) >> 20], 1u);
          }
        } else {
          for (int i = tid; i < L; i += kT) atomicAdd(&s.tau_bins[key_of(rowp.load1(i)) >> 20], 1u);
        }
        __syncthreads();
        // q = ceil(2k ns / L) sample keys above tau (integer arithmetic: FP64 is
        // a slow pipe on GB300 and every thread evaluates this)
        const int64_t want = (2 * static_cast<int64_t>(p.k) * ns + L - 1) / L;
        const uint32_t q = static_cast<uint32_t>(want < ns ? want : ns);
        tau = tau_from_bins(q > 0 ? q : 1u, s.tau_bins, s);
      }
      // 2. one streaming pass: compact the survivors (key >= tau); with two
      // CTAs, columns [0, h) and [h, L), h a multiple of 4 (16-byte loads)
      const int h = csize > 1 ? ((L + 7) >> 3) << 2 : L;
      const int c0 = rank == 0 ? 0 : h;
      const int c1 = rank == 0 ? h : L;
      const SrcGlobal<T> g{rowp.offset(c0), c1 - c0};
      uint32_t* const kw = s.data;
      uint32_t* const cw = s.data + kWarps * kWarpCap;
      if (rank == 0) {  // this CTA's shared memory, filled from the bottom
        if (tau > 0x80000000u) compact<true, false>(g, c0, tau, kw, cw, s.wsum, s.wmax);
        else compact<false, false>(g, c0, tau, kw, cw, s.wsum, s.wmax);
        if (csize == 1 && tid < kWarps) s.wsum[kWarps + tid] = 0;  // no top fill
      } else if constexpr (kCsize > 1) {  // rank 0's, through the cluster window, from the top
        uint32_t* const kr = s0.data;
        uint32_t* const cr = s0.data + kWarps * kWarpCap;
        if (tau > 0x80000000u)
          compact<true, true>(g, c0, tau, kr, cr, s0.wsum + kWarps, s0.wmax + kWarps);
        else
          compact<false, true>(g, c0, tau, kr, cr, s0.wsum + kWarps, s0.wmax + kWarps);
      }
      if constexpr (kCsize > 1) cg::this_cluster().sync();  // rank 1's survivors are in place
      else __syncthreads();
      if (rank == 0) {
        // one warp reduces the per-region counts and maxima (lane w: region w)
        // and shares them: every thread walking all regions took ~4 k cycles
        static_assert(kWarps == 32, "one lane per survivor region");
        if (tid < 32) {
          const uint32_t c = s.wsum[tid] + s.wsum[kWarps + tid];
          uint32_t m = s.wmax[tid];
          if (csize > 1) m = max(m, s.wmax[kWarps + tid]);
          const uint32_t tot = __reduce_add_sync(0xffffffffu, c);
          const uint32_t mx = __reduce_max_sync(0xffffffffu, m);
          const bool ov = __any_sync(0xffffffffu, c > static_cast<uint32_t>(kWarpCap));
          if (tid == 0) {
            s.stotal = tot;
            s.smax = mx;
            s.sover = ov ? 1u : 0u;
          }
        }
        __syncthreads();
        const uint32_t total = s.stotal, cmax = s.smax;
        const bool over = s.sover != 0;
        if (!over && total >= static_cast<uint32_t>(p.k)) {
          const SrcPairs sp{s.data, s.data + kWarps * kWarpCap, s.wsum};
          static_assert(kBins % kT == 0 && kBins <= 2048, "hist holds kBins bins");
          survivor_select_emit(sp, p.k, tau, cmax, p, row, s);
          done = true;
        } else if (tid == 0) {
          raise_error(p.err, kErrCapacity);
        }
      }
    }
    if (!done && rank == 0) {
      // full-row radix select (also the exact redo of a missed cutoff)
      if (!cutoff && L <= kStage) {
        for (int i4 = tid; 4 * i4 < L; i4 += kT) {
          const int e0 = 4 * i4;
          if (e0 + 3 < L) {
            const float4 v = rowp.load4(e0);
            *reinterpret_cast<uint4*>(s.data + e0) =
                make_uint4(key_of(v.x), key_of(v.y), key_of(v.z), key_of(v.w));
          } else {
            for (int j = e0; j < L; ++j) s.data[j] = key_of(rowp.load1(j));
          }
        }
        __syncthreads();
        const SrcStaged ss{s.data, L};
        const uint64_t thr = radix_select(ss, p.k, Sel{0, 0, 0u, 0u}, s);
        emit(ss, thr, p, row, s);
      } else {
        const SrcGlobal<T> g{rowp, L};
        const uint64_t thr = radix_select(g, p.k, Sel{0, 0, 0u, 0u}, s);
        emit(g, thr, p, row, s);
      }
    }
    __syncthreads();  // all emits done before the counter and the buffers are reused
    if constexpr (kCsize > 1) cg::this_cluster().sync();  // rank 0 is done with the regions rank 1 refills
    // both CTAs read the histogram before the syncs above: clear it for the
    // next use
    if (rank == 0 && hrow) clear_hist(hrow);
  }
}

}  // namespace

namespace {

template <class T>
cudaError_t launch_topk_t(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const size_t smem = sizeof(TkSmem) + 16;
  TkParams p{a.logits, a.ld,         a.row_len, a.R,          a.k,    a.col_blocks,
             a.nb,     a.block_size, a.out,     a.force_path, a.hist, dev.err_word};
  // Two CTAs per row while that leaves no row waiting for an SM and the rows
  // can be long enough for the halved streaming pass to repay the cluster's
  // costs: measured at 64 rows, k = 2048, the pair is ~2 us slower at 65536
  // columns, even at 98304 and ~2 us faster at 131072.
  const bool pair = 2 * a.R <= dev.sm_count && a.ld > 98304;
  cudaError_t e = cudaFuncSetAttribute(pair ? topk_kernel<2, T> : topk_kernel<1, T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (!pair) {
    const int grid = a.R < dev.sm_count ? a.R : dev.sm_count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<1, T>, p);
    return e == cudaSuccess ? cudaGetLastError() : e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.R);
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, topk_kernel<2, T>, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  return a.bf16 ? launch_topk_t<uint16_t>(a, dev, stream) : launch_topk_t<float>(a, dev, stream);
}

}  // namespace dsa
