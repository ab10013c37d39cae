// Internal constants shared by the host planners and the kernels of librx.
#pragma once
#include <stdint.h>

#include "rx.h"

namespace rx_internal {

// Decode: query rows (member requests x group heads) handled by one CTA.
constexpr int kDecodeRowsPerCta = 64;
// Decode: a segment chunk is at least this many keys (and at least 8 keys per
// query row, so partial results stay small next to the KV they summarise).
constexpr int kDecodeMinChunk = 512;
// Key tile of the attention kernels.
constexpr int kKeyTile = 64;

// Extend: query rows (query tokens x group heads) per CTA tile.
inline int extend_rows_per_tile(int head_dim) { return head_dim == 256 ? 64 : 128; }

rx_status set_error(rx_status s, const char* msg);

// Device-side helpers (kv_store.cu).
rx_status check_pool(const rx_pool_desc* pool, int32_t layer);
rx_status launch_status(const char* what);
int sm_count();
// Error words of the kernels of each file: bit 0 = slot out of range.
int32_t kv_store_error_flags(bool clear);
int32_t attention_error_flags(bool clear);

}  // namespace rx_internal
