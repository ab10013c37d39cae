// Internal constants shared by the host planners and the kernels of librx.
#pragma once
#include <stdint.h>

#include <cuda_runtime.h>

#include "rx.h"

namespace rx_internal {

// Decode work items: segments with at most decode_small_rows(head_dim) query
// rows (members x group heads) go to the warp role of the fused decode
// kernel (16 rows at head_dim 128; 8 at head_dim 256, where the O^T
// accumulators of 16 rows would not fit in the registers a warp of the
// 384-thread CTA has); larger ones are cut into member blocks of at most
// kDecodeTcRows rows for its tensor-core tiles.
inline int decode_small_rows(int head_dim) { return head_dim == 128 ? 16 : 8; }
constexpr int kDecodeTcRows = 128;
// Decode: segments of up to this many rows are split into warp-role items
// (member blocks of <= decode_small_rows rows) instead of a tensor-core tile.
constexpr int kDecodeSplitRows = 32;
inline int decode_rows_per_item(int /*head_dim*/) { return kDecodeTcRows; }
// Decode: a tensor-core chunk is at least kDecodeMinChunk keys and at least
// kDecodeKeysPerRow keys per query row of its segment (each tile CTA pays
// about 4 us of start-up and epilogue and writes 128 rows of partial
// results, so chunks are long); when that still gives more than
// kDecodeTcCap tile CTAs, every chunk is doubled until it does not (the
// tiles then run in about one wave beside the warp-role CTAs placed first).
constexpr int kDecodeMinChunk = 512;
constexpr int kDecodeKeysPerRow = 8;
constexpr int kDecodeTcCap = 128;
// Decode: a warp-role item's chunk is the largest of 128, 256, 512 and 1024
// keys that still leaves at least kDecodeUnitsPerWarp units (item x KV head)
// per warp-role warp of the GPU (152 SMs x 6 warps): long chunks spread a
// unit's start-up (work item, slot table, first K/V round trips) over more
// keys, short ones keep every warp busy when the batch has few private keys.
constexpr int kDecodeSmallChunkMin = 128;
constexpr int kDecodeSmallChunkMax = 1024;
constexpr int kDecodeWarpSlots = 152 * 6;
constexpr int kDecodeUnitsPerWarp = 2;

// Extend: query rows (query tokens x group heads) per CTA tile (the tcgen05
// tile kernel owns 128 TMEM lanes = 128 rows).
inline int extend_rows_per_tile(int /*head_dim*/) { return 128; }

rx_status set_error(rx_status s, const char* msg);

// Device-side helpers (kv_store.cu).
rx_status check_pool(const rx_pool_desc* pool, int32_t layer);
rx_status launch_status(const char* what);
int sm_count();
// Error words of the kernels of each file: bit 0 = slot out of range.
int32_t kv_store_error_flags(bool clear);
int32_t tc_error_flags(bool clear);
// One decode step in a single launch: the tensor-core tiles of the plan's
// large items and the warp-role units of its small items (attention_tc.cu).
// *unit_counter must be 0 at launch.  k_new / v_new / slots_new non-NULL:
// the warp owning a request's newest token stores it first.  Launched with
// programmatic stream serialization (the merge after it may launch early).
// early_inputs: the run's first step has completed when this kernel starts,
// so its tiles load queries and shared-segment keys (which no kernel of a
// run of decode steps writes) without griddepcontrol.wait, and wait only
// before writing partial results.
rx_status decode_fused(const rx_pool_desc* pool, int32_t layer, const void* d_q,
                       int32_t num_q_heads, const int32_t* d_req_to_token, int64_t row_stride,
                       const int32_t* d_work_small, int64_t n_small, const int32_t* d_work_tc,
                       int64_t n_tc, const int32_t* d_members, float scale, float* ws_o,
                       float* ws_lse, int32_t* unit_counter, int step, const void* k_new,
                       const void* v_new, const int32_t* slots_new, cudaStream_t stream,
                       bool early_inputs);
rx_status extend_attention_tc(const rx_pool_desc* pool, int32_t layer, const void* d_q,
                              int32_t num_q_heads, const int32_t* d_req_to_token,
                              int64_t row_stride, const int32_t* d_req_rows,
                              const int32_t* d_prefix_len, const int32_t* d_qo_indptr,
                              const int32_t* d_tile_indptr, int32_t R, int64_t num_tiles,
                              float scale, float* d_out, float* d_lse, cudaStream_t stream);

}  // namespace rx_internal
