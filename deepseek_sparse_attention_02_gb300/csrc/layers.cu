// A decode step over several DSA layers with the cross-layer selection
// schedules of the Multi-layer Indexer (MLI) abstract ("JEV Paper Radar"
// efficiency digest, 2026-11-04): IndexCache (only some layers run an indexer,
// the others reuse an earlier selection) and MLI (each layer attends the
// selection of the previous indexer layer, so its own indexer and top-k run on
// a second stream while its attention runs).  Host code only: the schedule is
// a sequence of the library's own entry points, ordered across the two
// streams by CUDA events.
//
// Buffers: one logits scratch (the indexers run one after another on the side
// stream) and two selection buffers used in turn by consecutive indexer
// layers.  The indexer of layer l writes the buffer the indexer before the
// previous one wrote; under MLI the last attention to read that selection is
// the one of the previous indexer layer (< l), and the side stream waits for
// the attention of layer l-1 before it starts, so it never overwrites a
// selection still being read.  Each buffer has its own event, so the main
// stream's wait for selection j never captures a later indexer's record.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "dsa.h"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status err(dsa_status st, const char* fmt, ...) {
  char msg[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  return static_cast<dsa_status>(set_last_error(st, msg));
}

// Events (no timing) of this host thread on each device: [0] attention done,
// [1] [2] selection buffer 0 / 1 written, [3] side stream drained.
struct ThreadEvents {
  cudaEvent_t ev[kMaxDevices][4] = {};
};
thread_local ThreadEvents t_events;

cudaError_t events_for_device(cudaEvent_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaEvent_t* ev = t_events.ev[dev];
  for (int i = 0; i < 4; ++i) {
    if (!ev[i]) {
      e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
  }
  *out = ev;
  return cudaSuccess;
}

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status dsa_layer_sources(const uint8_t* keep_indexer, int num_layers, int mli, int32_t* src) {
  using dsa::err;
  if (!keep_indexer || !src || num_layers < 1)
    return err(DSA_ERR_INVALID_ARG, "dsa_layer_sources: need keep_indexer, src, num_layers >= 1");
  if (!keep_indexer[0])
    return err(DSA_ERR_INVALID_ARG, "dsa_layer_sources: layer 0 must keep its indexer");
  int latest = -1;  // the latest indexer layer before the current one
  for (int l = 0; l < num_layers; ++l) {
    if (mli && l > 0) src[l] = latest;
    else src[l] = keep_indexer[l] ? l : latest;
    if (keep_indexer[l]) latest = l;
  }
  dsa::set_last_error(DSA_OK, "");
  return DSA_OK;
}

size_t dsa_decode_layers_workspace_size(int R, int64_t ld, int k) {
  if (R <= 0 || ld <= 0 || k <= 0) return 0;
  using dsa::align_up;
  return align_up(static_cast<size_t>(R) * ld * sizeof(float)) +
         2 * align_up(static_cast<size_t>(R) * k * sizeof(int32_t)) +
         align_up(dsa_sparse_mla_workspace_size(R, k));
}

dsa_status dsa_decode_layers(const dsa_layer* layers, int num_layers,
                             const uint8_t* keep_indexer, int mli, int64_t k_page_stride,
                             int64_t s_page_stride, int64_t kv_page_stride, int num_pages,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* ctx_len, const int32_t* row_len, int num_req,
                             int next_n, int k, float sm_scale, int64_t ld, void* workspace,
                             size_t workspace_bytes, void* stream, void* side_stream) {
  using dsa::aligned16;
  using dsa::err;
  const char* fn = "dsa_decode_layers";
  // ---- every check of the calls below, before anything is enqueued ----
  if (!layers || !keep_indexer || num_layers < 1 || !block_table || !ctx_len || !row_len)
    return err(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL or num_layers < 1", fn);
  if (!keep_indexer[0]) return err(DSA_ERR_INVALID_ARG, "%s: layer 0 must keep its indexer", fn);
  if (num_req < 0 || next_n < 1 || next_n > 65536 || num_pages < 1 || bt_stride < 1 || k < 1 ||
      k > DSA_MAX_TOPK || ld < 4 || ld % 4 || !(sm_scale > 0.f))
    return err(DSA_ERR_INVALID_ARG, "%s: bad sizes or scale", fn);
  if (num_req > 4096) return err(DSA_ERR_UNSUPPORTED, "%s: num_req > 4096", fn);
  const int64_t R64 = static_cast<int64_t>(num_req) * next_n;
  if (R64 * 64 > (1ll << 31) - 1 || R64 > (1 << 24) || ld > (1ll << 31) - 1)
    return err(DSA_ERR_UNSUPPORTED, "%s: too many rows or too long rows", fn);
  if (static_cast<int64_t>(num_pages) * 64 > (1ll << 31) - 1)
    return err(DSA_ERR_UNSUPPORTED, "%s: more than 2^31 cached rows", fn);
  if (k_page_stride < 64 * 128 || k_page_stride % 16 || s_page_stride < 256 ||
      s_page_stride % 16 || kv_page_stride != 64 * 576 * 2)
    return err(DSA_ERR_INVALID_ARG, "%s: bad page strides", fn);
  for (int l = 0; l < num_layers; ++l) {
    const dsa_layer& L = layers[l];
    if (!L.q || !L.kv_cache || !L.out || !aligned16(L.q) || !aligned16(L.kv_cache) ||
        !aligned16(L.out))
      return err(DSA_ERR_INVALID_ARG, "%s: layer %d: q, kv_cache, out must be 16-byte aligned", fn,
                 l);
    if (keep_indexer[l] && (!L.q_fp8 || !L.q_scale || !L.weights || !L.k_cache || !L.k_scale ||
                            !aligned16(L.q_fp8) || !aligned16(L.k_cache) || !aligned16(L.k_scale)))
      return err(DSA_ERR_INVALID_ARG,
                 "%s: layer %d keeps an indexer: q_fp8, q_scale, weights, k_cache, k_scale needed "
                 "(q_fp8, k_cache, k_scale 16-byte aligned)",
                 fn, l);
  }
  const int R = static_cast<int>(R64);
  if (R == 0) return static_cast<dsa_status>(dsa::set_last_error(DSA_OK, ""));
  const size_t need = dsa_decode_layers_workspace_size(R, ld, k);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return err(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, %zu given",
               fn, need, workspace_bytes);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* logits = reinterpret_cast<float*>(ws);
  ws += dsa::align_up(static_cast<size_t>(R) * ld * sizeof(float));
  int32_t* sel[2];
  for (int b = 0; b < 2; ++b) {
    sel[b] = reinterpret_cast<int32_t*>(ws);
    ws += dsa::align_up(static_cast<size_t>(R) * k * sizeof(int32_t));
  }
  void* mla_ws = ws;
  const size_t mla_bytes = dsa_sparse_mla_workspace_size(R, k);

  cudaStream_t main_s = static_cast<cudaStream_t>(stream);
  cudaStream_t side_s = side_stream ? static_cast<cudaStream_t>(side_stream) : main_s;
  const bool two = mli && side_s != main_s;
  cudaEvent_t* ev = nullptr;
  if (two) {
    const cudaError_t e = dsa::events_for_device(&ev);
    if (e != cudaSuccess) return err(DSA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  }
  auto cuda = [&](cudaError_t e) -> dsa_status {
    return e == cudaSuccess ? DSA_OK : err(DSA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  };

  // ---- the schedule ----
  int buf_of_latest = -1;  // selection buffer of the latest indexer layer
  int next_buf = 0;
  bool side_used = false;
  dsa_status st = DSA_OK;
  auto run_indexer = [&](int l, cudaStream_t s, int b) -> dsa_status {
    const dsa_layer& L = layers[l];
    dsa_status r = dsa_indexer_logits(L.q_fp8, L.q_scale, L.weights, L.k_cache, k_page_stride,
                                      L.k_scale, s_page_stride, num_pages, block_table, bt_stride,
                                      ctx_len, num_req, next_n, logits, ld, s);
    if (r != DSA_OK) return r;
    return dsa_topk(logits, ld, row_len, R, k, nullptr, 0, 0, sel[b], 0, s);
  };
  for (int l = 0; l < num_layers && st == DSA_OK; ++l) {
    const dsa_layer& L = layers[l];
    int src_buf;
    if (!mli || l == 0) {
      // the layer's own selection (when it keeps an indexer) precedes its attention
      if (keep_indexer[l]) {
        const int b = next_buf;
        next_buf ^= 1;
        if ((st = run_indexer(l, main_s, b)) != DSA_OK) break;
        buf_of_latest = b;
      }
      src_buf = buf_of_latest;
    } else {
      // attend the previous indexer layer's selection; this layer's indexer runs
      // on the side stream once the previous attention is done
      src_buf = buf_of_latest;
      if (two && side_used)  // the selection came from the side stream
        if ((st = cuda(cudaStreamWaitEvent(main_s, ev[1 + src_buf], 0))) != DSA_OK) break;
      if (keep_indexer[l]) {
        const int b = next_buf;
        next_buf ^= 1;
        if (two && (st = cuda(cudaStreamWaitEvent(side_s, ev[0], 0))) != DSA_OK) break;
        if ((st = run_indexer(l, side_s, b)) != DSA_OK) break;
        if (two && (st = cuda(cudaEventRecord(ev[1 + b], side_s))) != DSA_OK) break;
        side_used = true;
        buf_of_latest = b;
      }
    }
    if ((st = dsa_sparse_mla_decode(L.q, L.kv_cache, kv_page_stride, num_pages, block_table,
                                    bt_stride, num_req, next_n, sel[src_buf], k, sm_scale, L.out,
                                    L.lse, mla_ws, mla_bytes, main_s)) != DSA_OK)
      break;
    if (two && (st = cuda(cudaEventRecord(ev[0], main_s))) != DSA_OK) break;
  }
  if (two && side_used) {
    // the call ends on `stream`: it waits for the side stream's last top-k
    dsa_status s2 = cuda(cudaEventRecord(ev[3], side_s));
    if (s2 == DSA_OK) s2 = cuda(cudaStreamWaitEvent(main_s, ev[3], 0));
    if (st == DSA_OK) st = s2;
  }
  if (st == DSA_OK) dsa::set_last_error(DSA_OK, "");
  return st;
}

}  // extern "C"
