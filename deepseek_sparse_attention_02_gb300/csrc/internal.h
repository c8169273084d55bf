// Host-side launch interfaces between the C-ABI translation unit (dsa_api.cu)
// and the kernel translation units.  Arguments are validated by the caller.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
  uint32_t* err_word = nullptr;  // device address of this device's error word
};

// Launch attribute for programmatic dependent launch: the kernel may be
// scheduled while the previous kernel in the stream finishes; it waits for
// that kernel (griddepcontrol.wait) before it touches global memory.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Fills `info` for the current device.
cudaError_t current_device_info(DeviceInfo* info);

// Sets this host thread's dsa_last_error() message; returns `status`.
int set_last_error(int status, const char* msg);

// Encodes a CUtensorMap through the driver entry point (no libcuda link).
// dtype: 0 = uint8, 1 = bf16, 2 = 4-bit values, 16 packed in 8 bytes in
// global memory and padded to 16 bytes in shared memory (dims[0] counts the
// 4-bit values).  Returns false (and a message) on failure.
bool encode_tensor_map(void* map_out, int dtype, int rank, void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128,
                       char* msg, size_t msg_len);

struct IndexerArgs {
  const uint8_t* q;
  const float* q_scale;
  const float* w;
  const uint8_t* k_cache;
  int64_t k_page_stride;
  const uint8_t* k_scale;
  int64_t s_page_stride;
  int num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* ctx_len;
  int num_req;
  int next_n;               // rows per request, or (with cu_rows) the largest row count
  float* logits;
  int64_t ld;
  const int32_t* cu_rows = nullptr;  // varlen: request i's rows [cu_rows[i], cu_rows[i+1])
  const int32_t* bt_rows = nullptr;  // varlen: block-table row of request i
  int total_rows = 0;                // varlen: cu_rows[num_req]
  int bt_num_rows = 0;               // varlen: rows of the block table
  uint32_t* hist = nullptr;          // per-row score histograms [rows, 4096] (next_n <= 2)
};

cudaError_t launch_indexer(const IndexerArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                           char* msg, size_t msg_len);

struct TopkArgs {
  const void* logits;  // f32, or bf16 when bf16 != 0
  int64_t ld;
  const int32_t* row_len;
  int R;
  int k;
  const int32_t* col_blocks;
  int nb;
  int block_size;
  int32_t* out;
  int force_path;
  int bf16;
  uint32_t* hist = nullptr;  // per-row score histograms from the indexer; cleared on exit
};

cudaError_t launch_topk(const TopkArgs& a, const DeviceInfo& dev, cudaStream_t stream);

struct MlaArgs {
  const uint16_t* q;
  const uint16_t* kv;
  int64_t kv_page_stride;
  int num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int num_req;
  int next_n;
  const int32_t* idx;
  int k;
  float sm_scale;
  uint16_t* out;
  float* lse;
  void* ws;
  size_t ws_bytes;
  const int32_t* row_bt = nullptr;  // varlen: block-table row of each of the `rows` query rows
  int bt_num_rows = 0;
  int rows = 0;
};

// Split-K partials of R rows x k selections on a device with sm_count SMs
// (the split count follows the SM count).
size_t mla_workspace_size(int R, int k, int sm_count);
cudaError_t launch_sparse_mla(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// No-allocation variant: split-K scratch from a static device array.  The
// caller checks mla_workspace_size against mla_static_scratch_bytes first.
size_t mla_static_scratch_bytes();
cudaError_t launch_sparse_mla_static(const MlaArgs& a, const DeviceInfo& dev, cudaStream_t stream);

struct CandExpandArgs {
  const int32_t* cand;  // [R, nb_cand] candidate block ids
  int R;
  int nb;      // sparse blocks per row = nb_cand * expand
  int bs;      // sparse block size (the 64-token page)
  int expand;  // sparse blocks per candidate block
  const int32_t* ctx_len;
  int next_n;
  int32_t* sparse_indices;
  int32_t* end;
  void* schedule;
};

size_t candidate_schedule_size(int R);
cudaError_t launch_candidate_expand(const CandExpandArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream);

struct CandLogitsArgs {
  const uint8_t* q;
  const float* q_scale;
  const float* w;
  const uint8_t* k_fp4;
  int64_t k_page_stride;
  const uint8_t* k_sf;
  int64_t sf_page_stride;
  int num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int num_req;
  int next_n;
  const int32_t* sparse_indices;
  int nb;
  int bs;
  const int32_t* end;
  const void* schedule;
  float* logits;         // f32 output, or
  uint16_t* logits_bf16; // bf16 output (round to nearest even) when not null
  int64_t ld;
};

cudaError_t launch_candidate_logits(const CandLogitsArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream, char* msg, size_t msg_len);

}  // namespace dsa
