// S5: scatter new K/V rows into their pool slots, and the device
// req_to_token append.
//
// "SGLang: Structured LLM Programs for Efficient Inference", section "A quick
// recap of how an LLM generates text": every computed token's keys and values
// are stored in the KV cache; in decode each new token's own keys and values
// are appended.  "SGLang: the tree, and the language nobody remembers",
// section "Speculative decoding puts a tree inside the tree": the pool is
// addressed by KV indices (slots) that tree nodes hold.
//
// HBM-bound copy: each 16-byte chunk of a source row is read once
// (coalesced, contiguous) and written once to its slot's row (256 B or 512 B
// contiguous per (slot, head)).

#include <cuda_runtime.h>
#include <stdio.h>

#include <atomic>

#include "rx.h"
#include "rx_internal.h"

// Bit 0: rx_kv_store met a slot outside [1, num_slots); bit 4:
// rx_req_to_token_write met a row or position outside the table; bit 5:
// rx_kv_copy met a slot outside its pool.  The offending write is skipped.
// Read by rx_device_check().
static __device__ int32_t g_kv_store_error;

namespace {

__global__ void __launch_bounds__(256) kv_store_kernel(uint4* __restrict__ kdst,
                                                       uint4* __restrict__ vdst,
                                                       const int32_t* __restrict__ slots,
                                                       const uint4* __restrict__ ksrc,
                                                       const uint4* __restrict__ vsrc,
                                                       int64_t total_chunks, int hkv,
                                                       int chunks_per_row, int64_t head_stride,
                                                       int64_t num_slots) {
  const int64_t per_token = int64_t(hkv) * chunks_per_row;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < total_chunks;
       c += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = c / per_token;
    const int64_t rem = c - t * per_token;
    const int h = int(rem / chunks_per_row);
    const int j = int(rem - int64_t(h) * chunks_per_row);
    const int32_t slot = __ldg(slots + t);
    if (slot < 1 || slot >= num_slots) {  // never write outside the pool
      atomicOr(&g_kv_store_error, 1);
      continue;
    }
    const int64_t dst = h * head_stride + int64_t(slot) * chunks_per_row + j;
    const uint4 kv = __ldg(ksrc + c);
    const uint4 vv = __ldg(vsrc + c);
    kdst[dst] = kv;
    vdst[dst] = vv;
  }
}

// table[rows[i]][pos[i]] = slots[i]; an entry whose row is outside
// [0, num_rows) or whose position is outside [0, stride) is skipped and sets
// bit 4 of the error word, so a bad index never writes outside the table.
__global__ void r2t_write_kernel(int32_t* __restrict__ table, int64_t num_rows, int64_t stride,
                                 const int32_t* __restrict__ rows,
                                 const int32_t* __restrict__ pos,
                                 const int32_t* __restrict__ slots, int64_t n) {
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int32_t r = rows[i], p = pos[i];
  if (r < 0 || r >= num_rows || p < 0 || p >= stride) {
    atomicOr(&g_kv_store_error, 16);
    return;
  }
  table[int64_t(r) * stride + p] = slots[i];
}

// dst_pool[l][h][dst[i]][:] = src_pool[l][h][src[i]][:] for every layer and
// head: one 16-byte chunk per thread and iteration, chunks of a row on
// consecutive threads.  A slot outside [1, num_slots) of its pool skips the
// entry and sets bit 5 of the error word.  The pools may be the same (a move
// within the pool) or different (for example the device pool and a
// page-locked host pool the device reads and writes directly).
__global__ void __launch_bounds__(256) kv_copy_kernel(const uint4* __restrict__ src_k,
                                                      const uint4* __restrict__ src_v,
                                                      uint4* dst_k, uint4* dst_v,
                                                      const int32_t* __restrict__ src_slots,
                                                      const int32_t* __restrict__ dst_slots,
                                                      int64_t n, int L, int hkv, int cpr,
                                                      int64_t src_slots_n, int64_t dst_slots_n) {
  const int64_t per_entry = int64_t(L) * hkv * cpr;
  const int64_t total = n * per_entry;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += int64_t(gridDim.x) * blockDim.x) {
    const int64_t i = c / per_entry;
    int64_t rem = c - i * per_entry;
    const int64_t lh = rem / cpr;          // layer * hkv + head
    const int j = int(rem - lh * cpr);
    const int32_t s = __ldg(src_slots + i), t = __ldg(dst_slots + i);
    if (s < 1 || s >= src_slots_n || t < 1 || t >= dst_slots_n) {
      if (j == 0 && lh == 0) atomicOr(&g_kv_store_error, 32);
      continue;
    }
    const int64_t so = (lh * src_slots_n + s) * cpr + j;
    const int64_t to = (lh * dst_slots_n + t) * cpr + j;
    const uint4 kv = src_k[so];
    const uint4 vv = src_v[so];
    dst_k[to] = kv;
    dst_v[to] = vv;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace rx_internal {

rx_status check_pool(const rx_pool_desc* pool, int32_t layer) {
  if (!pool || !pool->k_pool || !pool->v_pool)
    return set_error(RX_ERR_INVALID, "pool descriptor or pool pointer is NULL");
  if (pool->head_dim != 128 && pool->head_dim != 256)
    return set_error(RX_ERR_INVALID, "head_dim must be 128 or 256");
  if (pool->num_kv_heads <= 0 || pool->num_layers <= 0 || pool->num_slots < 2)
    return set_error(RX_ERR_INVALID, "pool shape invalid");
  // the attention kernels address pool rows with 32-bit TMA coordinates
  if (int64_t(pool->num_layers) * pool->num_kv_heads * pool->num_slots > INT32_MAX)
    return set_error(RX_ERR_INVALID, "pool has 2^31 rows (layers x KV heads x slots) or more");
  if (layer < 0 || layer >= pool->num_layers)
    return set_error(RX_ERR_INVALID, "layer out of range");
  if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool))
    return set_error(RX_ERR_INVALID, "pool pointers must be 16-byte aligned");
  return RX_OK;
}

rx_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
    return set_error(RX_ERR_CUDA, buf);
  }
  return RX_OK;
}

int32_t kv_store_error_flags(bool clear) {
  int32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_kv_store_error, sizeof(v));
  if (clear && v) {
    int32_t z = 0;
    cudaMemcpyToSymbol(g_kv_store_error, &z, sizeof(z));
  }
  return v;
}

// SMs of the current device, queried once per device (152 if the query
// fails).
int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace rx_internal

extern "C" rx_status rx_kv_store(const rx_pool_desc* pool, int32_t layer, const int32_t* d_slots,
                                 const void* d_k, const void* d_v, int64_t T,
                                 rx_stream_t stream) {
  rx_status st = rx_internal::check_pool(pool, layer);
  if (st != RX_OK) return st;
  if (T < 0) return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_store: T < 0");
  if (T == 0) return RX_OK;
  if (!d_slots || !d_k || !d_v || !aligned16(d_k) || !aligned16(d_v))
    return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_store: NULL or misaligned input");
  const int cpr = pool->head_dim / 8;
  const int64_t head_stride = pool->num_slots * cpr;  // in 16-byte chunks
  const int64_t layer_off = int64_t(layer) * pool->num_kv_heads * head_stride;
  const int64_t total = T * pool->num_kv_heads * cpr;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(rx_internal::sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  kv_store_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<uint4*>(pool->k_pool) + layer_off,
      reinterpret_cast<uint4*>(pool->v_pool) + layer_off, d_slots,
      reinterpret_cast<const uint4*>(d_k), reinterpret_cast<const uint4*>(d_v), total,
      pool->num_kv_heads, cpr, head_stride, pool->num_slots);
  return rx_internal::launch_status("rx_kv_store");
}

extern "C" rx_status rx_req_to_token_write(int32_t* d_table, int64_t num_rows,
                                           int64_t row_stride, const int32_t* d_rows,
                                           const int32_t* d_pos, const int32_t* d_slots,
                                           int64_t n, rx_stream_t stream) {
  if (n < 0 || (n && (!d_table || !d_rows || !d_pos || !d_slots)) || row_stride <= 0 ||
      num_rows < 0)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_req_to_token_write: bad argument");
  if (n == 0) return RX_OK;
  r2t_write_kernel<<<unsigned((n + 255) / 256), 256, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(d_table, num_rows, row_stride,
                                                                d_rows, d_pos, d_slots, n);
  return rx_internal::launch_status("rx_req_to_token_write");
}

extern "C" rx_status rx_kv_copy(const rx_pool_desc* src, const rx_pool_desc* dst,
                                const int32_t* d_src_slots, const int32_t* d_dst_slots, int64_t n,
                                rx_stream_t stream) {
  rx_status st = rx_internal::check_pool(src, 0);
  if (st == RX_OK) st = rx_internal::check_pool(dst, 0);
  if (st != RX_OK) return st;
  if (src->num_layers != dst->num_layers || src->num_kv_heads != dst->num_kv_heads ||
      src->head_dim != dst->head_dim)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_copy: pools differ in shape");
  if (n < 0) return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_copy: n < 0");
  if (n == 0) return RX_OK;
  if (!d_src_slots || !d_dst_slots)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_copy: NULL slot list");
  // Every pool pointer must be one the device can reach: device (or
  // managed) memory as it is, page-locked host memory through its mapped
  // device address; pageable host memory is refused before any launch.
  void* ptr[4] = {src->k_pool, src->v_pool, dst->k_pool, dst->v_pool};
  for (void*& q : ptr) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
      cudaGetLastError();
      return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_copy: pool pointer unknown to CUDA");
    }
    if (at.type == cudaMemoryTypeHost) {
      if (!at.devicePointer)
        return rx_internal::set_error(RX_ERR_INVALID,
                                      "rx_kv_copy: host pool not mapped for device access");
      q = at.devicePointer;
    } else if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) {
      return rx_internal::set_error(RX_ERR_INVALID,
                                    "rx_kv_copy: pool must be device or page-locked host memory");
    }
    if (reinterpret_cast<uintptr_t>(q) & 15)
      return rx_internal::set_error(RX_ERR_INVALID, "rx_kv_copy: misaligned pool");
  }
  const int cpr = src->head_dim / 8;
  const int64_t total = n * src->num_layers * src->num_kv_heads * cpr;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(rx_internal::sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  kv_copy_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(ptr[0]), reinterpret_cast<const uint4*>(ptr[1]),
      reinterpret_cast<uint4*>(ptr[2]), reinterpret_cast<uint4*>(ptr[3]), d_src_slots,
      d_dst_slots, n, src->num_layers, src->num_kv_heads, cpr, src->num_slots, dst->num_slots);
  return rx_internal::launch_status("rx_kv_copy");
}

extern "C" rx_status rx_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return rx_internal::set_error(RX_ERR_INVALID, "rx_host_alloc: bad argument");
  *out = nullptr;
  // page-locked, mapped into the device address space (a host pool the
  // kernels read and write directly), usable from every device
  const cudaError_t e =
      cudaHostAlloc(out, bytes, cudaHostAllocPortable | cudaHostAllocMapped);
  if (e != cudaSuccess) {
    *out = nullptr;
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf), "rx_host_alloc: %zu bytes: %s", bytes, cudaGetErrorString(e));
    return rx_internal::set_error(RX_ERR_CUDA, buf);
  }
  return RX_OK;
}

extern "C" rx_status rx_host_free(void* p) {
  if (!p) return RX_OK;
  const cudaError_t e = cudaFreeHost(p);
  if (e != cudaSuccess) {
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf), "rx_host_free: %s", cudaGetErrorString(e));
    return rx_internal::set_error(RX_ERR_CUDA, buf);
  }
  return RX_OK;
}

extern "C" rx_status rx_device_check(int32_t* out_flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf), "rx_device_check: %s", cudaGetErrorString(e));
    return rx_internal::set_error(RX_ERR_CUDA, buf);
  }
  const int32_t tcf = rx_internal::tc_error_flags(true);
  int32_t f = rx_internal::kv_store_error_flags(true) | ((tcf & 7) << 1);
  if (out_flags) *out_flags = f;
  if (f)
    return rx_internal::set_error(RX_ERR_CUDA,
                                  (f & 8)    ? "rx_device_check: a tensor-core tile found its "
                                               "shared memory misaligned"
                                  : (f & 4)  ? "rx_device_check: a tensor-core kernel timed out "
                                               "waiting on a barrier"
                                  : (f & 16) ? "rx_device_check: a slot-table write met a row "
                                               "or position outside the table"
                                  : (f & 32) ? "rx_device_check: a KV copy met a slot outside "
                                               "its pool"
                                             : "rx_device_check: a kernel met a slot outside the pool");
  return RX_OK;
}

extern "C" const char* rx_build_info(void) {
  return "librx: host radix cache; kernels kv_store, extend/decode attention (sm_103a)";
}
