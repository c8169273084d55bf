// C ABI of the DSA decode path (declared in include/dsa.h): host-side argument
// validation, per-device state (SM count, device error word) and dispatch to
// the kernel launchers.  Every check runs before anything is enqueued; there is
// no fallback path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "dsa.h"
#include "internal.h"

namespace dsa {
namespace {

thread_local char g_msg[512] = "";

dsa_status fail(dsa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

dsa_status ok() {
  g_msg[0] = '\0';
  return DSA_OK;
}

// One error word per device.
__device__ uint32_t g_err_word;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int set_last_error(int status, const char* msg) {
  snprintf(g_msg, sizeof(g_msg), "%s", msg);
  return status;
}

cudaError_t current_device_info(DeviceInfo* info) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device != dev) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return e;
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_err_word);
    if (e != cudaSuccess) return e;
    d.sm_count = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.smem_optin = prop.sharedMemPerBlockOptin;
    d.err_word = static_cast<uint32_t*>(addr);
    d.device = dev;
  }
  *info = d;
  return cudaSuccess;
}

bool encode_tensor_map(void* map_out, int dtype, int rank, void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128,
                       char* msg, size_t msg_len) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  const CUtensorMapDataType dt = dtype == 0   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
  CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), dt, static_cast<cuuint32_t>(rank),
                        base, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return false;
  }
  return true;
}

namespace {

// Device checks shared by every entry point.
dsa_status device_ready(DeviceInfo* dev) {
  cudaError_t e = current_device_info(dev);
  if (e != cudaSuccess)
    return fail(DSA_ERR_CUDA, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (!(dev->cc_major == 10 && dev->cc_minor == 3))
    return fail(DSA_ERR_UNSUPPORTED,
                "this library is built for sm_103a (GB300); the current device is sm_%d%d",
                dev->cc_major, dev->cc_minor);
  return DSA_OK;
}

dsa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// dsa_indexer_logits / _varlen: the checks and the launch.  Without cu_rows
// every request has next_n rows; with it, entry i's rows are
// [cu_rows[i], cu_rows[i+1]) (at most next_n of them, total_rows in all) and
// it reads block-table row bt_rows[i] (or i).
dsa_status indexer_impl(const char* fn, const uint8_t* q_fp8, const float* q_scale,
                        const float* weights, const uint8_t* k_cache, int64_t k_page_stride,
                        const uint8_t* k_scale, int64_t s_page_stride, int num_pages,
                        const int32_t* block_table, int64_t bt_stride, const int32_t* ctx_len,
                        int num_req, int next_n, const int32_t* cu_rows, const int32_t* bt_rows,
                        int bt_num_rows, int total_rows, float* logits, int64_t ld,
                        uint32_t* hist, void* stream) {
  if (!q_fp8 || !q_scale || !weights || !k_cache || !k_scale || !block_table || !ctx_len ||
      !logits)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (num_req < 0 || next_n < 1 || next_n > 65536 || num_pages < 1 || bt_stride < 1 || ld < 4)
    return fail(DSA_ERR_INVALID_ARG,
                "%s: bad sizes (num_req=%d next_n=%d num_pages=%d bt_stride=%lld ld=%lld)", fn,
                num_req, next_n, num_pages, (long long)bt_stride, (long long)ld);
  const int64_t rows = cu_rows ? total_rows : static_cast<int64_t>(num_req) * next_n;
  if (rows * 64 > (1ll << 31) - 1) return fail(DSA_ERR_UNSUPPORTED, "%s: too many query rows", fn);
  if (num_req > 4096) return fail(DSA_ERR_UNSUPPORTED, "%s: num_req > 4096", fn);
  if (k_page_stride < 64 * 128 || k_page_stride % 16 || s_page_stride < 256 ||
      s_page_stride % 16)
    return fail(DSA_ERR_INVALID_ARG,
                "%s: page strides must cover the page payload and be multiples of 16 bytes", fn);
  if (!aligned16(k_cache) || !aligned16(k_scale) || !aligned16(q_fp8) || !aligned16(logits) ||
      ld % 4)
    return fail(DSA_ERR_INVALID_ARG,
                "%s: k_cache, k_scale, q_fp8 and logits must be 16-byte aligned, ld %% 4 == 0", fn);
  if (num_req == 0 || rows == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  IndexerArgs a{q_fp8,     q_scale,     weights,   k_cache, k_page_stride, k_scale, s_page_stride,
                num_pages, block_table, bt_stride, ctx_len, num_req,       next_n,  logits,
                ld};
  a.cu_rows = cu_rows;
  a.bt_rows = bt_rows;
  a.total_rows = static_cast<int>(rows);
  a.bt_num_rows = bt_num_rows;
  a.hist = hist;
  char msg[256] = "";
  cudaError_t e = launch_indexer(a, dev, static_cast<cudaStream_t>(stream), msg, sizeof(msg));
  if (e != cudaSuccess && msg[0]) return fail(DSA_ERR_UNSUPPORTED, "%s", msg);
  return cuda_status(e, fn);
}

// dsa_topk / dsa_topk_bf16: the checks and the launch, for f32 or bf16 scores.
dsa_status topk_impl(const char* fn, const void* logits, bool bf16, int64_t ld,
                     const int32_t* row_len, int R, int k, const int32_t* col_blocks, int nb,
                     int block_size, int32_t* out_idx, int force_path, uint32_t* hist,
                     void* stream) {
  if (!logits || !row_len || !out_idx)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (R < 0 || k < 1 || k > DSA_MAX_TOPK || ld < 4 || ld % 4 || !aligned16(logits))
    return fail(DSA_ERR_INVALID_ARG,
                "%s: need R >= 0, 1 <= k <= %d, ld %% 4 == 0, 16-byte aligned logits", fn,
                DSA_MAX_TOPK);
  if (ld > (1ll << 31) - 1) return fail(DSA_ERR_UNSUPPORTED, "%s: rows longer than 2^31", fn);
  if (col_blocks && (nb < 1 || block_size < 1))
    return fail(DSA_ERR_INVALID_ARG, "%s: col_blocks needs nb >= 1 and block_size >= 1", fn);
  if (force_path < 0 || force_path > 2)
    return fail(DSA_ERR_INVALID_ARG, "%s: force_path must be 0, 1 or 2", fn);
  if (R == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  TopkArgs a{logits, ld, row_len, R, k, col_blocks, nb, block_size, out_idx, force_path,
             bf16 ? 1 : 0};
  a.hist = hist;
  return cuda_status(launch_topk(a, dev, static_cast<cudaStream_t>(stream)), fn);
}

// dsa_candidate_logits / _bf16: the checks and the launch; exactly one of
// logits32 / logits16 is the output.
dsa_status cand_logits_impl(const char* fn, const uint8_t* q_fp8, const float* q_scale,
                            const float* weights, const uint8_t* k_fp4, int64_t k_page_stride,
                            const uint8_t* k_sf, int64_t sf_page_stride, int num_pages,
                            const int32_t* block_table, int64_t bt_stride, int num_req,
                            int next_n, const int32_t* sparse_indices, int nb, int block_size,
                            const int32_t* end, const void* schedule, size_t schedule_bytes,
                            float* logits32, uint16_t* logits16, int64_t ld, void* stream) {
  const void* logits = logits32 ? static_cast<const void*>(logits32) : logits16;
  if (!q_fp8 || !q_scale || !weights || !k_fp4 || !k_sf || !block_table || !sparse_indices ||
      !end || !schedule || !logits)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (num_req < 0 || next_n < 1 || num_pages < 1 || bt_stride < 1 || nb < 1)
    return fail(DSA_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (block_size != DSA_PAGE_TOKENS)
    return fail(DSA_ERR_UNSUPPORTED,
                "%s: the sparse block size must equal the %d-token page (got %d)", fn,
                DSA_PAGE_TOKENS, block_size);
  // the keys are read by a tensor copy of 4-bit elements: 32-byte aligned
  // base and page stride
  if (k_page_stride < 64 * 64 || k_page_stride % 32 || sf_page_stride < 256 ||
      sf_page_stride % 16 || reinterpret_cast<uintptr_t>(k_fp4) % 32 || !aligned16(k_sf) ||
      !aligned16(q_fp8) || !aligned16(logits) || ld % 4 ||
      ld < static_cast<int64_t>(nb) * block_size)
    return fail(DSA_ERR_INVALID_ARG,
                "%s: k_fp4 must be 32-byte aligned with k_page_stride %% 32 == 0, the other "
                "strides multiples of 16, buffers 16-byte aligned, ld >= nb*bs and ld %% 4 == 0",
                fn);
  const int64_t R64 = static_cast<int64_t>(num_req) * next_n;
  if (R64 > (1 << 20)) return fail(DSA_ERR_UNSUPPORTED, "%s: too many rows", fn);
  const int R = static_cast<int>(R64);
  if (schedule_bytes < candidate_schedule_size(R))
    return fail(DSA_ERR_WORKSPACE, "%s: schedule needs %zu bytes", fn,
                candidate_schedule_size(R));
  if (R == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  CandLogitsArgs a{q_fp8,          q_scale,   weights,     k_fp4,     k_page_stride, k_sf,
                   sf_page_stride, num_pages, block_table, bt_stride, num_req,       next_n,
                   sparse_indices, nb,        block_size,  end,       schedule,      logits32,
                   logits16,       ld};
  char msg[256] = "";
  cudaError_t e =
      launch_candidate_logits(a, dev, static_cast<cudaStream_t>(stream), msg, sizeof(msg));
  if (e != cudaSuccess && msg[0]) return fail(DSA_ERR_UNSUPPORTED, "%s", msg);
  return cuda_status(e, fn);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return 200; }

const char* dsa_last_error(void) { return g_msg; }

dsa_status dsa_get_device_error(void* stream, uint32_t* bits, int clear) {
  if (!bits) return fail(DSA_ERR_INVALID_ARG, "dsa_get_device_error: bits is NULL");
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return cuda_status(e, "dsa_get_device_error");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  e = cudaMemcpyAsync(&host, dev.err_word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    e = cudaMemsetAsync(dev.err_word, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_status(e, "dsa_get_device_error");
  *bits = host;
  return ok();
}

dsa_status dsa_indexer_logits(const uint8_t* q_fp8, const float* q_scale, const float* weights,
                              const uint8_t* k_cache, int64_t k_page_stride,
                              const uint8_t* k_scale, int64_t s_page_stride, int num_pages,
                              const int32_t* block_table, int64_t bt_stride,
                              const int32_t* ctx_len, int num_req, int next_n, float* logits,
                              int64_t ld, void* stream) {
  return dsa::indexer_impl("dsa_indexer_logits", q_fp8, q_scale, weights, k_cache, k_page_stride,
                           k_scale, s_page_stride, num_pages, block_table, bt_stride, ctx_len,
                           num_req, next_n, nullptr, nullptr, 0, 0, logits, ld, nullptr, stream);
}

dsa_status dsa_indexer_logits_varlen(const uint8_t* q_fp8, const float* q_scale,
                                     const float* weights, const uint8_t* k_cache,
                                     int64_t k_page_stride, const uint8_t* k_scale,
                                     int64_t s_page_stride, int num_pages,
                                     const int32_t* block_table, int64_t bt_stride,
                                     int bt_num_rows, const int32_t* bt_rows,
                                     const int32_t* ctx_len, const int32_t* cu_rows,
                                     int num_entries, int max_rows, int total_rows,
                                     float* logits, int64_t ld, void* stream) {
  const char* fn = "dsa_indexer_logits_varlen";
  if (!cu_rows) return fail(DSA_ERR_INVALID_ARG, "%s: cu_rows is NULL", fn);
  if (max_rows < 1 || max_rows > 65536 || total_rows < 0 || bt_num_rows < 1 ||
      (!bt_rows && bt_num_rows < num_entries))
    return fail(DSA_ERR_INVALID_ARG,
                "%s: need 1 <= max_rows <= 65536, total_rows >= 0, bt_num_rows >= 1 (and >= "
                "num_entries without bt_rows)",
                fn);
  return dsa::indexer_impl(fn, q_fp8, q_scale, weights, k_cache, k_page_stride, k_scale,
                           s_page_stride, num_pages, block_table, bt_stride, ctx_len, num_entries,
                           max_rows, cu_rows, bt_rows, bt_num_rows, total_rows, logits, ld,
                           nullptr, stream);
}

dsa_status dsa_topk(const float* logits, int64_t ld, const int32_t* row_len, int R, int k,
                    const int32_t* col_blocks, int nb, int block_size, int32_t* out_idx,
                    int force_path, void* stream) {
  return dsa::topk_impl("dsa_topk", logits, false, ld, row_len, R, k, col_blocks, nb, block_size,
                        out_idx, force_path, nullptr, stream);
}

dsa_status dsa_topk_bf16(const uint16_t* logits, int64_t ld, const int32_t* row_len, int R, int k,
                         const int32_t* col_blocks, int nb, int block_size, int32_t* out_idx,
                         int force_path, void* stream) {
  return dsa::topk_impl("dsa_topk_bf16", logits, true, ld, row_len, R, k, col_blocks, nb,
                        block_size, out_idx, force_path, nullptr, stream);
}

size_t dsa_score_hist_size(int R) {
  if (R <= 0) return 0;
  return static_cast<size_t>(R) * DSA_HIST_BINS * sizeof(uint32_t);
}

dsa_status dsa_indexer_logits_hist(const uint8_t* q_fp8, const float* q_scale,
                                   const float* weights, const uint8_t* k_cache,
                                   int64_t k_page_stride, const uint8_t* k_scale,
                                   int64_t s_page_stride, int num_pages,
                                   const int32_t* block_table, int64_t bt_stride,
                                   const int32_t* ctx_len, int num_req, int next_n, float* logits,
                                   int64_t ld, uint32_t* hist, void* stream) {
  const char* fn = "dsa_indexer_logits_hist";
  if (!hist || !aligned16(hist))
    return fail(DSA_ERR_INVALID_ARG, "%s: hist must be a 16-byte aligned device buffer", fn);
  if (next_n > 2)
    return fail(DSA_ERR_UNSUPPORTED,
                "%s: score histograms are built for decode (next_n <= 2), got next_n %d", fn,
                next_n);
  return dsa::indexer_impl(fn, q_fp8, q_scale, weights, k_cache, k_page_stride, k_scale,
                           s_page_stride, num_pages, block_table, bt_stride, ctx_len, num_req,
                           next_n, nullptr, nullptr, 0, 0, logits, ld, hist, stream);
}

dsa_status dsa_topk_hist(const float* logits, int64_t ld, const int32_t* row_len, int R, int k,
                         uint32_t* hist, int32_t* out_idx, int force_path, void* stream) {
  const char* fn = "dsa_topk_hist";
  if (!hist || !aligned16(hist))
    return fail(DSA_ERR_INVALID_ARG, "%s: hist must be a 16-byte aligned device buffer", fn);
  return dsa::topk_impl(fn, logits, false, ld, row_len, R, k, nullptr, 0, 0, out_idx, force_path,
                        hist, stream);
}

// The SM count the sparse MLA's work split is sized for: the current
// device's, or GB300's 152 when no device can be queried (a size asked for on
// a machine without a GPU).
static int mla_sm_count() {
  DeviceInfo dev;
  if (current_device_info(&dev) == cudaSuccess && dev.sm_count > 0) return dev.sm_count;
  cudaGetLastError();  // the failed query leaves no sticky error for later calls
  return 152;
}

size_t dsa_sparse_mla_workspace_size(int R, int k) {
  if (R <= 0 || k <= 0) return 0;
  return mla_workspace_size(R, k, mla_sm_count());
}

dsa_status dsa_sparse_mla_decode(const uint16_t* q, const uint16_t* kv_cache,
                                 int64_t kv_page_stride, int num_pages,
                                 const int32_t* block_table, int64_t bt_stride, int num_req,
                                 int next_n, const int32_t* idx, int k, float sm_scale,
                                 uint16_t* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const char* fn = "dsa_sparse_mla_decode";
  if (!q || !kv_cache || !block_table || !idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (num_req < 0 || next_n < 1 || num_pages < 1 || bt_stride < 1 || k < 1 ||
      k > DSA_MAX_TOPK || !(sm_scale > 0.f))
    return fail(DSA_ERR_INVALID_ARG, "%s: bad sizes or scale", fn);
  if (kv_page_stride != 64 * 576 * 2 || !aligned16(kv_cache) || !aligned16(q) ||
      !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG,
                "%s: latent pages must be contiguous (kv_page_stride == 73728); q, kv and out "
                "16-byte aligned",
                fn);
  if (static_cast<int64_t>(num_pages) * 64 > (1ll << 31) - 1)
    return fail(DSA_ERR_UNSUPPORTED, "%s: more than 2^31 cached latent rows", fn);
  const int64_t R64 = static_cast<int64_t>(num_req) * next_n;
  if (R64 > (1 << 24)) return fail(DSA_ERR_UNSUPPORTED, "%s: too many rows", fn);
  const int R = static_cast<int>(R64);
  if (R == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  const size_t need = mla_workspace_size(R, k, dev.sm_count);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace_bytes);
  MlaArgs a{q,   kv_cache, kv_page_stride, num_pages, block_table, bt_stride, num_req, next_n,
            idx, k,        sm_scale,       out,       lse,         workspace, workspace_bytes};
  return cuda_status(launch_sparse_mla(a, dev, static_cast<cudaStream_t>(stream)), fn);
}

size_t dsa_candidate_schedule_size(int R) {
  if (R <= 0) return 0;
  return candidate_schedule_size(R);
}

dsa_status dsa_candidate_expand(const int32_t* cand, int R, int nb, int block_size,
                                const int32_t* ctx_len, int next_n, int32_t* sparse_indices,
                                int32_t* end, void* schedule, size_t schedule_bytes,
                                void* stream) {
  const char* fn = "dsa_candidate_expand";
  if (!cand || !ctx_len || !sparse_indices || !end || !schedule)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (R < 0 || nb < 1 || next_n < 1 || (R % next_n) != 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: need nb >= 1, next_n >= 1, R %% next_n == 0", fn);
  if (block_size < DSA_PAGE_TOKENS || block_size % DSA_PAGE_TOKENS ||
      block_size > 64 * DSA_PAGE_TOKENS)
    return fail(DSA_ERR_UNSUPPORTED,
                "%s: candidate_block_size must be 1..64 times the %d-token page (got %d)", fn,
                DSA_PAGE_TOKENS, block_size);
  const int expand = block_size / DSA_PAGE_TOKENS;
  if (static_cast<int64_t>(nb) * expand > 4096)
    return fail(DSA_ERR_UNSUPPORTED, "%s: more than 4096 sparse blocks per row", fn);
  if (schedule_bytes < candidate_schedule_size(R))
    return fail(DSA_ERR_WORKSPACE, "%s: schedule needs %zu bytes", fn,
                candidate_schedule_size(R));
  if (R == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  CandExpandArgs a{cand,    R,      nb * expand,    DSA_PAGE_TOKENS, expand,
                   ctx_len, next_n, sparse_indices, end,             schedule};
  return cuda_status(launch_candidate_expand(a, dev, static_cast<cudaStream_t>(stream)), fn);
}

dsa_status dsa_candidate_logits(const uint8_t* q_fp8, const float* q_scale, const float* weights,
                                const uint8_t* k_fp4, int64_t k_page_stride, const uint8_t* k_sf,
                                int64_t sf_page_stride, int num_pages,
                                const int32_t* block_table, int64_t bt_stride, int num_req,
                                int next_n, const int32_t* sparse_indices, int nb,
                                int block_size, const int32_t* end, const void* schedule,
                                size_t schedule_bytes, float* logits, int64_t ld, void* stream) {
  return dsa::cand_logits_impl("dsa_candidate_logits", q_fp8, q_scale, weights, k_fp4,
                               k_page_stride, k_sf, sf_page_stride, num_pages, block_table,
                               bt_stride, num_req, next_n, sparse_indices, nb, block_size, end,
                               schedule, schedule_bytes, logits, nullptr, ld, stream);
}

dsa_status dsa_candidate_logits_bf16(const uint8_t* q_fp8, const float* q_scale,
                                     const float* weights, const uint8_t* k_fp4,
                                     int64_t k_page_stride, const uint8_t* k_sf,
                                     int64_t sf_page_stride, int num_pages,
                                     const int32_t* block_table, int64_t bt_stride, int num_req,
                                     int next_n, const int32_t* sparse_indices, int nb,
                                     int block_size, const int32_t* end, const void* schedule,
                                     size_t schedule_bytes, uint16_t* logits, int64_t ld,
                                     void* stream) {
  return dsa::cand_logits_impl("dsa_candidate_logits_bf16", q_fp8, q_scale, weights, k_fp4,
                               k_page_stride, k_sf, sf_page_stride, num_pages, block_table,
                               bt_stride, num_req, next_n, sparse_indices, nb, block_size, end,
                               schedule, schedule_bytes, nullptr, logits, ld, stream);
}

dsa_status dsa_sparse_mla_decode_varlen(const uint16_t* q, const uint16_t* kv_cache,
                                        int64_t kv_page_stride, int num_pages,
                                        const int32_t* block_table, int64_t bt_stride,
                                        int bt_num_rows, const int32_t* row_bt, int R,
                                        const int32_t* idx, int k, float sm_scale, uint16_t* out,
                                        float* lse, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  const char* fn = "dsa_sparse_mla_decode_varlen";
  if (!q || !kv_cache || !block_table || !row_bt || !idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (R < 0 || bt_num_rows < 1 || num_pages < 1 || bt_stride < 1 || k < 1 ||
      k > DSA_MAX_TOPK || !(sm_scale > 0.f))
    return fail(DSA_ERR_INVALID_ARG, "%s: bad sizes or scale", fn);
  if (kv_page_stride != 64 * 576 * 2 || !aligned16(kv_cache) || !aligned16(q) ||
      !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG,
                "%s: latent pages must be contiguous (kv_page_stride == 73728); q, kv and out "
                "16-byte aligned",
                fn);
  if (static_cast<int64_t>(num_pages) * 64 > (1ll << 31) - 1)
    return fail(DSA_ERR_UNSUPPORTED, "%s: more than 2^31 cached latent rows", fn);
  if (R > (1 << 24)) return fail(DSA_ERR_UNSUPPORTED, "%s: too many rows", fn);
  if (R == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  const size_t need = mla_workspace_size(R, k, dev.sm_count);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace_bytes);
  MlaArgs a{q,   kv_cache, kv_page_stride, num_pages, block_table, bt_stride, 1,         1,
            idx, k,        sm_scale,       out,       lse,         workspace, workspace_bytes};
  a.row_bt = row_bt;
  a.bt_num_rows = bt_num_rows;
  a.rows = R;
  return cuda_status(launch_sparse_mla(a, dev, static_cast<cudaStream_t>(stream)), fn);
}

size_t dsa_sparse_mla_static_scratch_bytes(void) { return mla_static_scratch_bytes(); }

dsa_status dsa_sparse_mla_decode_static(const uint16_t* q, const uint16_t* kv_cache,
                                        int64_t kv_page_stride, int num_pages,
                                        const int32_t* block_table, int64_t bt_stride,
                                        int num_req, int next_n, const int32_t* idx, int k,
                                        float sm_scale, uint16_t* out, float* lse,
                                        void* stream) {
  const char* fn = "dsa_sparse_mla_decode_static";
  if (!q || !kv_cache || !block_table || !idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (num_req < 0 || next_n < 1 || num_pages < 1 || bt_stride < 1 || k < 1 ||
      k > DSA_MAX_TOPK || !(sm_scale > 0.f))
    return fail(DSA_ERR_INVALID_ARG, "%s: bad sizes or scale", fn);
  if (kv_page_stride != 64 * 576 * 2 || !aligned16(kv_cache) || !aligned16(q) ||
      !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG,
                "%s: latent pages must be contiguous (kv_page_stride == 73728); q, kv and out "
                "16-byte aligned",
                fn);
  if (static_cast<int64_t>(num_pages) * 64 > (1ll << 31) - 1)
    return fail(DSA_ERR_UNSUPPORTED, "%s: more than 2^31 cached latent rows", fn);
  const int64_t R64 = static_cast<int64_t>(num_req) * next_n;
  if (R64 > (1 << 24)) return fail(DSA_ERR_UNSUPPORTED, "%s: too many rows", fn);
  if (R64 == 0) return ok();
  DeviceInfo dev;
  dsa_status st = device_ready(&dev);
  if (st != DSA_OK) return st;
  const size_t need = mla_workspace_size(static_cast<int>(R64), k, dev.sm_count);
  if (need > mla_static_scratch_bytes())
    return fail(DSA_ERR_UNSUPPORTED,
                "%s: this batch needs %zu bytes of split-K scratch but the static scratch holds "
                "%zu; call dsa_sparse_mla_decode with a workspace instead",
                fn, need, mla_static_scratch_bytes());
  MlaArgs a{q,   kv_cache, kv_page_stride, num_pages, block_table, bt_stride, num_req, next_n,
            idx, k,        sm_scale,       out,       lse,         nullptr,   0};
  return cuda_status(launch_sparse_mla_static(a, dev, static_cast<cudaStream_t>(stream)), fn);
}

}  // extern "C"
