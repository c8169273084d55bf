// Prefill in chunks (the vLLM "sparse_indexer" page: the prefill chunker
// budgets the f32 logits [rows, seq_len] of a chunk, every row counted at
// least min_split_seq_len wide; a chunk's rows carry per-row K ranges and may
// come from several requests).
//
// dsa_prefill_chunk_plan (host) splits a batch's query rows into such chunks.
// A chunk is then run as "entries": each piece (request b, rows [j0, j1) of
// its n_b) is an entry of j1 - j0 rows whose last row sees ctx_b - (n_b - j1)
// tokens, read through block-table row b (dsa_indexer_logits_varlen,
// dsa_sparse_mla_decode_varlen); dsa_varlen_row_lengths writes the rows' key
// counts for dsa_topk.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "dsa.h"
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

dsa_status err(dsa_status st, const char* fmt, ...) {
  char msg[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  return static_cast<dsa_status>(set_last_error(st, msg));
}

// One CTA per entry: row cu[e] + j of entry e sees ctx[e] - (n_e - 1 - j)
// tokens.  An entry whose row range is reversed or outside [0, total] writes
// nothing and sets the bad-index bit.
__global__ void varlen_row_lengths_kernel(const int32_t* ctx, const int32_t* cu, int total,
                                          int32_t* row_len, uint32_t* err) {
  const int e = blockIdx.x;
  const int a = cu[e], b = cu[e + 1];
  if (a < 0 || b < a || b > total) {
    if (threadIdx.x == 0) raise_error(err, kErrBadIndex);
    return;
  }
  const int n = b - a;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int L = ctx[e] - (n - 1 - j);
    row_len[a + j] = L > 0 ? L : 0;
  }
}

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status dsa_prefill_chunk_plan(const int32_t* q_len, const int32_t* ctx_len, int num_req,
                                  int64_t budget_bytes, int64_t min_cols, int32_t* pieces,
                                  int max_pieces, int* num_pieces) {
  using dsa::err;
  const char* fn = "dsa_prefill_chunk_plan";
  if (!q_len || !ctx_len || !pieces || !num_pieces || num_req < 0 || max_pieces < 0 ||
      budget_bytes < 1 || min_cols < 0)
    return err(DSA_ERR_INVALID_ARG, "%s: bad arguments", fn);
  int np = 0, chunk = 0;
  int64_t rows = 0, width = 0;  // the current chunk's rows and widest row
  for (int b = 0; b < num_req; ++b) {
    if (q_len[b] < 0 || ctx_len[b] < 0)
      return err(DSA_ERR_INVALID_ARG, "%s: negative length for request %d", fn, b);
    int64_t w = ctx_len[b] > min_cols ? ctx_len[b] : min_cols;
    w = (w + 3) / 4 * 4;  // the logits row stride is a multiple of 4
    for (int j = 0; j < q_len[b]; ++j) {
      const int64_t wide = width > w ? width : w;
      if (rows > 0 && (rows + 1) * wide * 4 > budget_bytes) {  // the row opens a new chunk
        ++chunk;
        rows = 0;
        width = 0;
      }
      int32_t* last = np > 0 ? pieces + 4 * (np - 1) : nullptr;
      if (last && last[0] == chunk && last[1] == b) {
        last[3] = j + 1;
      } else {
        if (np == max_pieces)
          return err(DSA_ERR_WORKSPACE, "%s: more than %d pieces", fn, max_pieces);
        int32_t* pc = pieces + 4 * np++;
        pc[0] = chunk;
        pc[1] = b;
        pc[2] = j;
        pc[3] = j + 1;
      }
      ++rows;
      if (w > width) width = w;
    }
  }
  *num_pieces = np;
  dsa::set_last_error(DSA_OK, "");
  return DSA_OK;
}

dsa_status dsa_varlen_row_lengths(const int32_t* ctx_len, const int32_t* cu_rows, int num_entries,
                                  int total_rows, int32_t* row_len, void* stream) {
  using dsa::err;
  const char* fn = "dsa_varlen_row_lengths";
  if (!ctx_len || !cu_rows || !row_len || num_entries < 0 || total_rows < 0)
    return err(DSA_ERR_INVALID_ARG, "%s: bad arguments", fn);
  if (num_entries == 0) return static_cast<dsa_status>(dsa::set_last_error(DSA_OK, ""));
  dsa::DeviceInfo dev;
  cudaError_t e = dsa::current_device_info(&dev);
  if (e == cudaSuccess) {
    dsa::varlen_row_lengths_kernel<<<num_entries, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        ctx_len, cu_rows, total_rows, row_len, dev.err_word);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return err(DSA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  dsa::set_last_error(DSA_OK, "");
  return DSA_OK;
}

}  // extern "C"
