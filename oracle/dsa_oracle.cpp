// DeepSeek Sparse Attention decode path -- fp64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
// CUDA library is checked against.  Only the test-suite, the smoke check and the
// CPU-baseline leg of the benchmark may load it; the product path never does.
// It shares no code, header, table or helper with the CUDA sources.
//
// Every value is decoded exactly to double and every formula is evaluated as
// written, with no blocking, fusion or reordering:
//
//  * Indexer score, Eq. (1) of "DeepSeek V3.2-Exp support" (llama.cpp issue
//    16331, section "1. Architecture"):
//        I_{t,s} = sum_j w_{t,j} * ReLU(q_{t,j} . k_s)
//    with q_{t,j} = sq_{t,j} * dec_e4m3(q'_{t,j}) (per-head q scale) and
//    k_s = s_s * dec_e4m3(k'_s) (per-token key scale of the FP8 key cache,
//    "an extra cache to store a 128-element k_s value for each token").
//  * Candidate-block scores: the same sum over the tokens of the candidate
//    blocks only ("vLLM sparse_indexer" API page, module docstring; the
//    "[DSA] Wire DeepGEMM sparse MQA logits" item of the RepoJournal digest),
//    with MXFP4 keys: e2m1 elements times a UE8M0 scale per 32 elements
//    (sparse_indexer builder: "UE8M0-packed granularity-32 scales").
//  * Fine-grained token selection: Top-k of I_{t,:} by a full sort
//    (score descending, then token index ascending), Eq. (2) context.
//  * Sparse attention, Eq. (2): softmax attention of the query over the
//    selected latents c_s only; the value is the first 512 of the 576
//    elements ("512 or 576 element vectors", same issue).
//
// Parity pins for every function live in tests/test_oracle_*.py.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- decoding --

// FP8 E4M3 ("fn" variant: no infinities, S.1111.111 is NaN): sign bit, 4-bit
// exponent with bias 7, 3-bit mantissa; exponent field 0 is subnormal.
double dec_e4m3(uint8_t b, bool* is_nan) {
  const int sign = (b >> 7) & 1;
  const int e = (b >> 3) & 0xF;
  const int m = b & 7;
  if (e == 0xF && m == 7) {
    *is_nan = true;
    return std::numeric_limits<double>::quiet_NaN();
  }
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(m), -9);  // m/8 * 2^(1-7)
  } else {
    mag = std::ldexp(8.0 + m, e - 7 - 3);  // (1 + m/8) * 2^(e-7)
  }
  return sign ? -mag : mag;
}

// FP4 E2M1 (OCP MX): sign bit, 2-bit exponent with bias 1, 1-bit mantissa.
double dec_e2m1(uint8_t nib) {
  const int sign = (nib >> 3) & 1;
  const int e = (nib >> 1) & 3;
  const int m = nib & 1;
  double mag;
  if (e == 0) {
    mag = 0.5 * m;
  } else {
    mag = std::ldexp(2.0 + m, e - 1 - 1);  // (1 + m/2) * 2^(e-1)
  }
  return sign ? -mag : mag;
}

// UE8M0 (OCP MX scale): unsigned 8-bit exponent, value 2^(e-127); 0xFF is NaN.
double dec_ue8m0(uint8_t e, bool* is_nan) {
  if (e == 0xFF) {
    *is_nan = true;
    return std::numeric_limits<double>::quiet_NaN();
  }
  return std::ldexp(1.0, static_cast<int>(e) - 127);
}

// bfloat16: the upper half of an IEEE binary32.
double dec_bf16(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

float load_f32(const uint8_t* p) {
  float f;
  std::memcpy(&f, p, 4);
  return f;
}

// Runs fn(i) for i in [0, n) on up to nthreads std::threads.
template <typename F>
void parallel_for(int n, int nthreads, F fn) {
  if (nthreads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (;;) {
      const int i = next.fetch_add(1);
      if (i >= n) return;
      fn(i);
    }
  };
  const int t = std::min(nthreads, n);
  std::vector<std::thread> pool;
  pool.reserve(t);
  for (int i = 0; i < t; ++i) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

// Row r = req * next_n + j sees ctx_len[req] - (next_n - 1 - j) tokens: the
// next_n query rows of one request are consecutive draft positions and the
// cache already holds every one of them.
int64_t row_len(const int32_t* ctx_len, int next_n, int r) {
  const int req = r / next_n;
  const int j = r % next_n;
  const int64_t L = static_cast<int64_t>(ctx_len[req]) - (next_n - 1 - j);
  return L < 0 ? 0 : L;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------- plain decoders --

int orc_decode_e4m3(const uint8_t* in, int64_t n, double* out) {
  int nans = 0;
  for (int64_t i = 0; i < n; ++i) {
    bool bad = false;
    out[i] = dec_e4m3(in[i], &bad);
    nans += bad;
  }
  return nans;
}

// n_elems e2m1 values packed two per byte: element 2i is the low nibble of
// byte i, element 2i+1 the high nibble.
int orc_decode_e2m1(const uint8_t* packed, int64_t n_elems, double* out) {
  for (int64_t i = 0; i < n_elems; ++i) {
    const uint8_t byte = packed[i / 2];
    out[i] = dec_e2m1((i & 1) ? (byte >> 4) : (byte & 0xF));
  }
  return 0;
}

int orc_decode_ue8m0(const uint8_t* in, int64_t n, double* out) {
  int nans = 0;
  for (int64_t i = 0; i < n; ++i) {
    bool bad = false;
    out[i] = dec_ue8m0(in[i], &bad);
    nans += bad;
  }
  return nans;
}

int orc_decode_bf16(const uint16_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec_bf16(in[i]);
  return 0;
}

// ------------------------------------------------------- dense indexer, Eq.1 --
//
// q       [R, H, D] e4m3 codes; q_scale [R, H] f32 (> 0); w [R, H] f32.
// Key cache page p: D-byte e4m3 key of slot i at k_cache + p*k_page_stride +
// i*D; its f32 scale at k_scale + p*s_page_stride + 4*i (both in bytes).
// Token t of request req lives in page block_table[req*bt_stride + t/page_tokens],
// slot t % page_tokens.
// For each row rows[i] this writes logits[i*ld + t] = I and mag[i*ld + t] =
// sum_j |w_j| ReLU(q_j . k_t) (the scale against which a rounding error in the
// sum is judged) for t < L_r.  Returns the number of NaN codes met (0 = ok).
int orc_indexer_logits(const uint8_t* q, const float* q_scale, const float* w,
                       const uint8_t* k_cache, int64_t k_page_stride,
                       const uint8_t* k_scale, int64_t s_page_stride,
                       int page_tokens, const int32_t* block_table,
                       int64_t bt_stride, const int32_t* ctx_len, int num_req,
                       int next_n, int H, int D, const int32_t* rows,
                       int nrows, double* logits, double* mag, int64_t ld,
                       int nthreads) {
  (void)num_req;
  std::atomic<int> nans{0};
  parallel_for(nrows, nthreads, [&](int i) {
    const int r = rows[i];
    const int req = r / next_n;
    const int64_t L = row_len(ctx_len, next_n, r);
    bool bad = false;
    std::vector<double> qd(static_cast<size_t>(H) * D);
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d)
        qd[h * D + d] = static_cast<double>(q_scale[r * H + h]) *
                        dec_e4m3(q[(static_cast<int64_t>(r) * H + h) * D + d], &bad);
    std::vector<double> kd(D);
    for (int64_t t = 0; t < L; ++t) {
      const int64_t page = block_table[req * bt_stride + t / page_tokens];
      const int64_t slot = t % page_tokens;
      const uint8_t* kp = k_cache + page * k_page_stride + slot * D;
      const double s = load_f32(k_scale + page * s_page_stride + 4 * slot);
      for (int d = 0; d < D; ++d) kd[d] = s * dec_e4m3(kp[d], &bad);
      double I = 0.0, A = 0.0;
      for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[h * D + d] * kd[d];
        const double relu = dot > 0.0 ? dot : 0.0;
        const double wh = w[r * H + h];
        I += wh * relu;
        A += std::fabs(wh) * relu;
      }
      logits[i * ld + t] = I;
      if (mag) mag[i * ld + t] = A;
    }
    if (bad) nans.fetch_add(1);
  });
  return nans.load();
}

// ---------------------------------------------------- candidate expansion --
//
// cand [R, nb]: candidate block ids of each row, as a source layer publishes
// them.  Writes sparse_indices [R, nb] = the ids sorted ascending and end[r] =
// the number of sparse columns c (c in [0, nb*bs)) whose token
// tok(c) = sparse_indices[r][c/bs]*bs + c%bs is a valid position of the row
// (0 <= tok < L_r).
int orc_candidate_expand(const int32_t* cand, int R, int nb, int bs,
                         const int32_t* ctx_len, int next_n,
                         int32_t* sparse_indices, int32_t* end) {
  for (int r = 0; r < R; ++r) {
    std::vector<int32_t> ids(cand + static_cast<int64_t>(r) * nb,
                             cand + static_cast<int64_t>(r + 1) * nb);
    std::sort(ids.begin(), ids.end());
    const int64_t L = row_len(ctx_len, next_n, r);
    int64_t cnt = 0;
    for (int c = 0; c < nb * bs; ++c) {
      const int64_t tok = static_cast<int64_t>(ids[c / bs]) * bs + c % bs;
      if (tok >= 0 && tok < L) ++cnt;
    }
    std::copy(ids.begin(), ids.end(), sparse_indices + static_cast<int64_t>(r) * nb);
    end[r] = static_cast<int32_t>(cnt);
  }
  return 0;
}

// ------------------------------------------- candidate (sparse MQA) logits --
//
// Keys are MXFP4: page p holds, for slot i, D/2 packed e2m1 bytes at
// k_fp4 + p*k_page_stride + i*D/2 and D/32 UE8M0 bytes at
// k_sf + p*sf_page_stride + i*D/32 (byte g scales elements 32g..32g+31).
// The per-token FP8 key scale has no counterpart here: s_t = 1.
// Column c < end[r] scores token tok(c) as in orc_candidate_expand.
int orc_candidate_logits(const uint8_t* q, const float* q_scale, const float* w,
                         const uint8_t* k_fp4, int64_t k_page_stride,
                         const uint8_t* k_sf, int64_t sf_page_stride,
                         int page_tokens, const int32_t* block_table,
                         int64_t bt_stride, int next_n, int H, int D,
                         const int32_t* sparse_indices, int nb, int bs,
                         const int32_t* end, const int32_t* rows, int nrows,
                         double* logits, double* mag, int64_t ld, int nthreads) {
  std::atomic<int> nans{0};
  parallel_for(nrows, nthreads, [&](int i) {
    const int r = rows[i];
    const int req = r / next_n;
    bool bad = false;
    std::vector<double> qd(static_cast<size_t>(H) * D);
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d)
        qd[h * D + d] = static_cast<double>(q_scale[r * H + h]) *
                        dec_e4m3(q[(static_cast<int64_t>(r) * H + h) * D + d], &bad);
    std::vector<double> kd(D);
    for (int64_t c = 0; c < end[r]; ++c) {
      const int64_t tok =
          static_cast<int64_t>(sparse_indices[static_cast<int64_t>(r) * nb + c / bs]) * bs +
          c % bs;
      const int64_t page = block_table[req * bt_stride + tok / page_tokens];
      const int64_t slot = tok % page_tokens;
      const uint8_t* kp = k_fp4 + page * k_page_stride + slot * (D / 2);
      const uint8_t* sp = k_sf + page * sf_page_stride + slot * (D / 32);
      for (int d = 0; d < D; ++d) {
        const uint8_t byte = kp[d / 2];
        const double v = dec_e2m1((d & 1) ? (byte >> 4) : (byte & 0xF));
        kd[d] = v * dec_ue8m0(sp[d / 32], &bad);
      }
      double I = 0.0, A = 0.0;
      for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[h * D + d] * kd[d];
        const double relu = dot > 0.0 ? dot : 0.0;
        const double wh = w[r * H + h];
        I += wh * relu;
        A += std::fabs(wh) * relu;
      }
      logits[i * ld + c] = I;
      if (mag) mag[i * ld + c] = A;
    }
    if (bad) nans.fetch_add(1);
  });
  return nans.load();
}

// ------------------------------------------------------------------ top-k --
//
// For each of nrows rows: order the columns [0, len[i]) by score descending,
// ties by column ascending, keep the first min(k, len) and pad with -1.
// If col_blocks is given ([nrows, nb]), column c is reported as token
// col_blocks[i][c/bs]*bs + c%bs.
int orc_topk(const double* scores, int64_t ld, const int32_t* len, int nrows,
             int k, const int32_t* col_blocks, int nb, int bs, int32_t* out,
             int nthreads) {
  parallel_for(nrows, nthreads, [&](int i) {
    const int64_t L = len[i] < 0 ? 0 : len[i];
    std::vector<int64_t> order(L);
    for (int64_t c = 0; c < L; ++c) order[c] = c;
    const double* s = scores + i * ld;
    std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
      if (s[a] != s[b]) return s[a] > s[b];
      return a < b;
    });
    for (int j = 0; j < k; ++j) {
      int64_t v = -1;
      if (j < L) {
        v = order[j];
        if (col_blocks)
          v = static_cast<int64_t>(col_blocks[static_cast<int64_t>(i) * nb + v / bs]) * bs +
              v % bs;
      }
      out[static_cast<int64_t>(i) * k + j] = static_cast<int32_t>(v);
    }
  });
  return 0;
}

// ----------------------------------------------------- sparse MLA, Eq. (2) --
//
// q [R, Hq, Dqk] bf16; latent cache page p, slot i: Dqk bf16 at
// kv + (p*kv_page_stride + i*Dqk) elements.  Row r belongs to request
// r / next_n.  idx [R, k]: selected token positions, -1 = none.
// For head g: z_j = scale * q_g . c_j over the valid selected j,
// p = softmax(z), O_g = sum_j p_j c_j[0:Dv], lse_g = log sum_j exp(z_j).
// A row with no valid index gives O = 0 and lse = -inf.
int orc_sparse_mla(const uint16_t* q, const uint16_t* kv, int64_t kv_page_stride,
                   int page_tokens, const int32_t* block_table, int64_t bt_stride,
                   int next_n, const int32_t* idx, int k, int Hq, int Dqk, int Dv,
                   double scale, const int32_t* rows, int nrows, double* out,
                   double* lse, int nthreads) {
  parallel_for(nrows, nthreads, [&](int i) {
    const int r = rows[i];
    const int req = r / next_n;
    std::vector<const uint16_t*> sel;
    for (int j = 0; j < k; ++j) {
      const int32_t t = idx[static_cast<int64_t>(r) * k + j];
      if (t < 0) continue;
      const int64_t page = block_table[req * bt_stride + t / page_tokens];
      sel.push_back(kv + page * kv_page_stride + static_cast<int64_t>(t % page_tokens) * Dqk);
    }
    const size_t n = sel.size();
    std::vector<double> c(n * Dqk);
    for (size_t j = 0; j < n; ++j)
      for (int d = 0; d < Dqk; ++d) c[j * Dqk + d] = dec_bf16(sel[j][d]);
    std::vector<double> z(n);
    for (int g = 0; g < Hq; ++g) {
      const uint16_t* qg = q + (static_cast<int64_t>(r) * Hq + g) * Dqk;
      double* o = out + (static_cast<int64_t>(i) * Hq + g) * Dv;
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      if (n == 0) {
        lse[static_cast<int64_t>(i) * Hq + g] = -std::numeric_limits<double>::infinity();
        continue;
      }
      double m = -std::numeric_limits<double>::infinity();
      for (size_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < Dqk; ++d) dot += dec_bf16(qg[d]) * c[j * Dqk + d];
        z[j] = scale * dot;
        m = std::max(m, z[j]);
      }
      double sum = 0.0;
      for (size_t j = 0; j < n; ++j) sum += std::exp(z[j] - m);
      for (size_t j = 0; j < n; ++j) {
        const double p = std::exp(z[j] - m) / sum;
        for (int d = 0; d < Dv; ++d) o[d] += p * c[j * Dqk + d];
      }
      lse[static_cast<int64_t>(i) * Hq + g] = m + std::log(sum);
    }
  });
  return 0;
}

int orc_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n == 0 ? 1 : static_cast<int>(n);
}

}  // extern "C"
