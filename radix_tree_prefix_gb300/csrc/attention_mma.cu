// S6-S9: the C entry points of extend and decode attention over the radix KV
// pool and the log-sum-exp merge of decode partials.  The attention itself
// runs on the tcgen05 kernels of attention_tc.cu.
//
// What is computed ("SGLang: Structured LLM Programs for Efficient
// Inference", sections "A quick recap of how an LLM generates text" and "How
// RadixAttention reuses past work"): each query attends, with softmax, over
// the keys of its request up to and including itself; keys of a reused prefix
// are read from the pool slots the radix cache handed out, exactly as if they
// had just been computed.  Query head h reads KV head h / (Hq/Hkv).  Decode
// splits each request's context into the plan's segments (a tree segment
// shared by several requests is read once for all of them); each segment
// chunk yields a partial (o, lse) per query row, and the merge combines a
// request's partials: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "ptx_util.cuh"
#include "rx.h"
#include "rx_internal.h"

namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;

// One warp per (request, query head): lse = log sum_s exp(lse_s),
// o = sum_s exp(lse_s - lse) o_s over the request's partial entries.  The
// plan's part lists are read before the wait for the decode kernel; after it,
// lane i reads part i's lse while the first eight parts' rows are already in
// flight, so a request with up to eight parts costs one round trip to memory.
// Partials are read through L2 (they were written by the previous kernel).
// Block 0 also resets the decode kernel's work counter for the next step.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const int32_t* __restrict__ indptr,
                                                        const int32_t* __restrict__ parts,
                                                        const float* __restrict__ ws_o,
                                                        const float* __restrict__ ws_lse,
                                                        int hq, int B, float* __restrict__ out,
                                                        float* __restrict__ lse_out,
                                                        int32_t* __restrict__ counter,
                                                        int late_trigger) {
  constexpr int V = D / 128;  // float4 per lane
  constexpr int CH = 8;       // part rows loaded together
  // launched after the decode kernel with programmatic stream serialization:
  // let the next step's kernel start launching, then wait for the partials.
  // late_trigger: the next kernel may launch only once this one has waited,
  // i.e. once the decode kernel before it has completed.
  if (!late_trigger) rxk::griddep_launch_dependents();
  const int gw = int(blockIdx.x) * 8 + int(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const bool active = gw < B * hq;
  const int b = active ? gw / hq : 0;
  const int h = active ? gw - b * hq : 0;
  const int p0 = active ? indptr[b] : 0;
  const int n = active ? indptr[b + 1] - p0 : 0;
  int64_t e = lane < n ? int64_t(parts[p0 + lane]) * hq + h : 0;
  rxk::griddep_wait();
  if (late_trigger) rxk::griddep_launch_dependents();
  if (counter && blockIdx.x == 0 && threadIdx.x == 0) *counter = 0;
  if (!active) return;
  const float4* o4 = reinterpret_cast<const float4*>(ws_o);
  float4 x[CH][V];
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int64_t ek = __shfl_sync(0xffffffffu, e, k);
    if (k < n)
#pragma unroll
      for (int v = 0; v < V; ++v) x[k][v] = __ldcg(o4 + ek * (D / 4) + v * 32 + lane);
  }
  float li = lane < n ? __ldcg(ws_lse + e) : -INFINITY;
  float m = li;
  for (int i = lane + 32; i < n; i += 32)
    m = fmaxf(m, __ldcg(ws_lse + int64_t(parts[p0 + i]) * hq + h));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float w = li == -INFINITY ? 0.f : rxk::fast_exp2((li - m) * kLog2e);
  float sum = w;
  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const float wk = __shfl_sync(0xffffffffu, w, k);
    if (k < n)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        acc[v].x += wk * x[k][v].x;
        acc[v].y += wk * x[k][v].y;
        acc[v].z += wk * x[k][v].z;
        acc[v].w += wk * x[k][v].w;
      }
  }
  // parts beyond the first eight (long contexts split into many chunks)
  for (int base = 0; base < n; base += 32) {
    if (base > 0) {
      const int i = base + lane;
      e = i < n ? int64_t(parts[p0 + i]) * hq + h : 0;
      const float lj = i < n ? __ldcg(ws_lse + e) : -INFINITY;
      w = lj == -INFINITY ? 0.f : rxk::fast_exp2((lj - m) * kLog2e);
      sum += w;
    }
    const int j0 = base == 0 ? CH : 0;
    const int cnt = min(32, n - base);
    for (int j = j0; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const int64_t ej = __shfl_sync(0xffffffffu, e, j);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const float4 y = __ldcg(o4 + ej * (D / 4) + v * 32 + lane);
        acc[v].x += wj * y.x;
        acc[v].y += wj * y.y;
        acc[v].z += wj * y.z;
        acc[v].w += wj * y.w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  float4* dst = reinterpret_cast<float4*>(out + (int64_t(b) * hq + h) * D);
#pragma unroll
  for (int v = 0; v < V; ++v)
    dst[v * 32 + lane] = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
  if (lane == 0) lse_out[int64_t(b) * hq + h] = m + logf(sum);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" rx_status rx_extend_attention(const rx_pool_desc* pool, int32_t layer,
                                         const void* d_q, int32_t num_q_heads,
                                         const int32_t* d_req_to_token, int64_t row_stride,
                                         const int32_t* d_req_rows, const int32_t* d_prefix_len,
                                         const int32_t* d_qo_indptr,
                                         const int32_t* d_tile_indptr, int32_t R,
                                         int64_t num_tiles, float scale, float* d_out,
                                         float* d_lse, rx_stream_t stream) {
  rx_status st = rx_internal::check_pool(pool, layer);
  if (st != RX_OK) return st;
  if (num_q_heads <= 0 || num_q_heads % pool->num_kv_heads != 0)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_extend_attention: Hq % Hkv != 0");
  if (R < 0 || num_tiles < 0 || num_tiles * pool->num_kv_heads > INT32_MAX)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_extend_attention: bad R or num_tiles");
  if (R == 0 || num_tiles == 0) return RX_OK;
  if (!d_q || !d_req_to_token || !d_req_rows || !d_prefix_len || !d_qo_indptr ||
      !d_tile_indptr || !d_out || !d_lse || !aligned16(d_q) || !aligned16(d_out))
    return rx_internal::set_error(RX_ERR_INVALID, "rx_extend_attention: NULL or misaligned");
  return rx_internal::extend_attention_tc(pool, layer, d_q, num_q_heads, d_req_to_token,
                                         row_stride, d_req_rows, d_prefix_len, d_qo_indptr,
                                         d_tile_indptr, R, num_tiles, scale, d_out, d_lse,
                                         reinterpret_cast<cudaStream_t>(stream));
}

namespace {

rx_status decode_attention_impl(const rx_pool_desc* pool, int32_t layer, const void* d_q,
                                int32_t num_q_heads, const int32_t* d_req_to_token,
                                int64_t row_stride, const int32_t* d_plan,
                                const rx_decode_plan_info* info, int32_t B, float scale,
                                float* d_out, float* d_lse, void* d_workspace,
                                size_t workspace_bytes, cudaStream_t s, bool first_call,
                                int step, const void* k_new = nullptr,
                                const void* v_new = nullptr,
                                const int32_t* slots_new = nullptr,
                                int32_t* counter_at = nullptr, bool early_inputs = false,
                                bool late_trigger = false) {
  rx_status st = rx_internal::check_pool(pool, layer);
  if (st != RX_OK) return st;
  if (!info || num_q_heads <= 0 || num_q_heads % pool->num_kv_heads != 0 || B < 0)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_attention: bad argument");
  if (B == 0) return RX_OK;
  if (int64_t(workspace_bytes) < info->workspace_bytes || !d_workspace ||
      !aligned16(d_workspace))
    return rx_internal::set_error(RX_ERR_INVALID,
                                  "rx_decode_attention: workspace missing, small or misaligned");
  if (!d_q || !d_req_to_token || !d_plan || !d_out || !d_lse || !aligned16(d_q) ||
      !aligned16(d_out) || info->n_work > INT32_MAX)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_attention: NULL or misaligned");
  const int D = pool->head_dim;
  const int32_t* work = d_plan + info->off_work;
  const int32_t* members = d_plan + info->off_members;
  const int64_t o_bytes = info->n_parts * num_q_heads * int64_t(D) * 4;
  float* ws_o = static_cast<float*>(d_workspace);
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(d_workspace) + ((o_bytes + 255) / 256) * 256);
  const int64_t l_bytes = info->n_parts * num_q_heads * 4;
  int32_t* counter = counter_at ? counter_at
                                : reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws_lse) +
                                                             ((l_bytes + 255) / 256) * 256);
  // the work counter of the decode kernel is 0 at every launch: zeroed here
  // once per call, reset by each merge after that
  if (first_call && cudaMemsetAsync(counter, 0, sizeof(int32_t), s) != cudaSuccess)
    return rx_internal::launch_status("decode counter reset");
  if (info->n_work > 0) {
    const int64_t n_small = info->n_work - info->n_work_tc;
    st = rx_internal::decode_fused(pool, layer, d_q, num_q_heads, d_req_to_token, row_stride, work,
                                   n_small, work + n_small * RX_WORK_WORDS, info->n_work_tc,
                                   members, scale, ws_o, ws_lse, counter, step, k_new, v_new,
                                   slots_new, s, early_inputs);
    if (st != RX_OK) return st;
  }
  // The merge may launch while the decode kernel before it still runs (it
  // waits on the device for that kernel's results), so its launch latency is
  // hidden.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned((int64_t(B) * num_q_heads + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t* indptr = d_plan + info->off_req_part_indptr;
  const int32_t* parts = d_plan + info->off_req_parts;
  const float* wo = ws_o;
  const float* wl = ws_lse;
  if (D == 128)
    cudaLaunchKernelEx(&cfg, lse_merge_kernel<128>, indptr, parts, wo, wl, int(num_q_heads),
                       int(B), d_out, d_lse, counter, late_trigger ? 1 : 0);
  else
    cudaLaunchKernelEx(&cfg, lse_merge_kernel<256>, indptr, parts, wo, wl, int(num_q_heads),
                       int(B), d_out, d_lse, counter, late_trigger ? 1 : 0);
  return rx_internal::launch_status("decode merge");
}

}  // namespace

extern "C" rx_status rx_decode_attention(const rx_pool_desc* pool, int32_t layer,
                                         const void* d_q, int32_t num_q_heads,
                                         const int32_t* d_req_to_token, int64_t row_stride,
                                         const int32_t* d_plan, const rx_decode_plan_info* info,
                                         int32_t B, float scale, float* d_out, float* d_lse,
                                         void* d_workspace, size_t workspace_bytes,
                                         rx_stream_t stream) {
  return decode_attention_impl(pool, layer, d_q, num_q_heads, d_req_to_token, row_stride, d_plan,
                               info, B, scale, d_out, d_lse, d_workspace, workspace_bytes,
                               reinterpret_cast<cudaStream_t>(stream), true, 0);
}

extern "C" rx_status rx_verify_attention(const rx_pool_desc* pool, int32_t layer,
                                         const void* d_q, int32_t num_q_heads,
                                         const int32_t* d_req_to_token, int64_t row_stride,
                                         const int32_t* d_plan, const rx_decode_plan_info* info,
                                         int32_t N, float scale, float* d_out, float* d_lse,
                                         void* d_workspace, size_t workspace_bytes,
                                         rx_stream_t stream) {
  // every draft token is one query of the plan; its row holds the context
  // and its root path, so the decode kernels apply the tree mask
  return decode_attention_impl(pool, layer, d_q, num_q_heads, d_req_to_token, row_stride, d_plan,
                               info, N, scale, d_out, d_lse, d_workspace, workspace_bytes,
                               reinterpret_cast<cudaStream_t>(stream), true, 0);
}

extern "C" rx_status rx_decode_steps(const rx_pool_desc* pool, int32_t layer, int32_t num_q_heads,
                                     const int32_t* d_req_to_token, int64_t row_stride,
                                     const rx_decode_step* steps, int32_t n_steps, int32_t B,
                                     float scale, void* d_workspace, size_t workspace_bytes,
                                     rx_stream_t stream) {
  if (n_steps < 0 || (n_steps && !steps))
    return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_steps: bad step list");
  rx_status r = rx_internal::check_pool(pool, layer);
  if (r != RX_OK) return r;
  if (num_q_heads <= 0 || num_q_heads % pool->num_kv_heads != 0)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_steps: Hq % Hkv != 0");
  const int G = num_q_heads / pool->num_kv_heads;
  // A run of steps whose new tokens all lie in private tails: every step has
  // its own work counter (zeroed here at once, after the largest step's
  // partial results), step 0's merge lets the next kernel launch only after
  // step 0 has completed, and later steps' tiles then read their queries and
  // the shared segments (no kernel of the run writes those) without waiting
  // for the step before; only their partial writes wait for its merge.
  bool early = n_steps >= 2 && B > 0 && G <= rx_internal::decode_small_rows(pool->head_dim);
  int64_t region = 0;
  for (int32_t i = 0; early && i < n_steps; ++i) {
    const rx_decode_plan_info* inf = steps[i].info;
    if (!inf || inf->tails_private != 1) {
      early = false;
      break;
    }
    const int64_t o = inf->n_parts * num_q_heads * int64_t(pool->head_dim) * 4;
    const int64_t l = inf->n_parts * num_q_heads * 4;
    region = std::max<int64_t>(region, (o + 255) / 256 * 256 + (l + 255) / 256 * 256);
  }
  if (early && (!d_workspace || int64_t(workspace_bytes) < region + 4 * int64_t(n_steps)))
    early = false;
  int32_t* counters =
      early ? reinterpret_cast<int32_t*>(static_cast<char*>(d_workspace) + region) : nullptr;
  if (early && cudaMemsetAsync(counters, 0, 4 * size_t(n_steps),
                               reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return rx_internal::launch_status("decode counters reset");
  for (int32_t i = 0; i < n_steps; ++i) {
    const rx_decode_step& st = steps[i];
    // every step's new token is the end of a growing private tail: the decode
    // kernel's warp role stores it itself
    const bool fused = B > 0 && G <= rx_internal::decode_small_rows(pool->head_dim) && st.info &&
                       st.info->tails_private == 1;
    if (!fused) {
      r = rx_kv_store(pool, layer, st.d_slots, st.d_k, st.d_v, B, stream);
      if (r != RX_OK) return r;
    } else if (!st.d_k || !st.d_v || !st.d_slots || (reinterpret_cast<uintptr_t>(st.d_k) & 15) ||
               (reinterpret_cast<uintptr_t>(st.d_v) & 15)) {
      return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_steps: NULL or misaligned K/V");
    }
    r = decode_attention_impl(pool, layer, st.d_q, num_q_heads, d_req_to_token, row_stride,
                              st.d_plan, st.info, B, scale, st.d_out, st.d_lse, d_workspace,
                              workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                              i == 0 && !early, st.step, fused ? st.d_k : nullptr,
                              fused ? st.d_v : nullptr, fused ? st.d_slots : nullptr,
                              early ? counters + i : nullptr, early && i > 0, early && i == 0);
    if (r != RX_OK) return r;
  }
  return RX_OK;
}

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot provide device memory.
//
// rx_decode_attention needs a caller-owned scratch buffer for its partial
// results.  Some callers have no way to get one: a host process whose device
// memory is entirely reserved up front by its own pool, or a plugin that is
// handed a stream and pointers but no allocator.  This entry point keeps the
// scratch in a fixed array that lives in the library's device image instead:
// it exists on every GPU that loads the library, for as long as the process
// runs, and is RX_DECODE_STATIC_SCRATCH_BYTES long.  It runs exactly the same
// kernels as rx_decode_attention.
static __device__ __align__(256) unsigned char g_decode_static_scratch[RX_DECODE_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kStaticMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_scratch_ptr[kStaticMaxDevices];
}  // namespace

extern "C" rx_status rx_decode_attention_static(const rx_pool_desc* pool, int32_t layer,
                                                const void* d_q, int32_t num_q_heads,
                                                const int32_t* d_req_to_token, int64_t row_stride,
                                                const int32_t* d_plan,
                                                const rx_decode_plan_info* info, int32_t B,
                                                float scale, float* d_out, float* d_lse,
                                                rx_stream_t stream) {
  if (!info) return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_attention_static: no plan info");
  if (info->workspace_bytes > int64_t(RX_DECODE_STATIC_SCRATCH_BYTES)) {
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf),
             "rx_decode_attention_static: the plan needs %lld bytes of scratch, the static "
             "scratch holds %lld; use rx_decode_attention with a larger buffer",
             (long long)info->workspace_bytes, (long long)RX_DECODE_STATIC_SCRATCH_BYTES);
    return rx_internal::set_error(RX_ERR_INVALID, buf);
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices)
    return rx_internal::set_error(RX_ERR_CUDA, "rx_decode_attention_static: no usable current device");
  void* scratch = nullptr;
  {
    // First call on this device: look up the device address of the array
    // (a host-side reference to it is not a device pointer).
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_scratch_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
      if (e != cudaSuccess || !p) {
        static thread_local char buf[256];
        snprintf(buf, sizeof(buf), "rx_decode_attention_static: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(e));
        return rx_internal::set_error(RX_ERR_CUDA, buf);
      }
      g_static_scratch_ptr[dev] = p;
    }
    scratch = g_static_scratch_ptr[dev];
  }
  return decode_attention_impl(pool, layer, d_q, num_q_heads, d_req_to_token, row_stride, d_plan,
                               info, B, scale, d_out, d_lse, scratch,
                               size_t(RX_DECODE_STATIC_SCRATCH_BYTES),
                               reinterpret_cast<cudaStream_t>(stream), true, 0);
}

extern "C" rx_status rx_extend_batches(const rx_pool_desc* pool, int32_t layer,
                                       int32_t num_q_heads, const rx_extend_batch* batches,
                                       int32_t n, float scale, const rx_event_t* events,
                                       rx_stream_t stream) {
  if (n < 0 || (n && !batches))
    return rx_internal::set_error(RX_ERR_INVALID, "rx_extend_batches: bad batch list");
  rx_status r = rx_internal::check_pool(pool, layer);
  if (r != RX_OK) return r;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto mark = [&](int32_t i, int k) -> rx_status {
    if (!events) return RX_OK;
    if (cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[4 * int64_t(i) + k]), s) !=
        cudaSuccess)
      return rx_internal::launch_status("rx_extend_batches: event record");
    return RX_OK;
  };
  // batch i + 1 reads the KV that batch i stored (its prefix may end inside
  // batch i's tokens): the launches stay in batch order on one stream
  for (int32_t i = 0; i < n; ++i) {
    const rx_extend_batch& b = batches[i];
    if ((r = mark(i, 0)) != RX_OK) return r;
    r = rx_kv_store(pool, layer, b.d_new_slots, b.d_k, b.d_v, b.n_new, stream);
    if (r != RX_OK) return r;
    if ((r = mark(i, 1)) != RX_OK || (r = mark(i, 2)) != RX_OK) return r;
    r = rx_extend_attention(pool, layer, b.d_q, num_q_heads, b.d_req_to_token, b.row_stride,
                            b.d_req_rows, b.d_prefix_len, b.d_qo_indptr, b.d_tile_indptr, b.R,
                            b.num_tiles, scale, b.d_out, b.d_lse, stream);
    if (r != RX_OK) return r;
    if ((r = mark(i, 3)) != RX_OK) return r;
  }
  return RX_OK;
}

extern "C" rx_status rx_events_create(int32_t n, rx_event_t* out) {
  if (n < 0 || (n && !out)) return rx_internal::set_error(RX_ERR_INVALID, "rx_events_create");
  for (int32_t i = 0; i < n; ++i) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (int32_t j = 0; j < i; ++j) cudaEventDestroy(reinterpret_cast<cudaEvent_t>(out[j]));
      return rx_internal::launch_status("rx_events_create");
    }
    out[i] = reinterpret_cast<rx_event_t>(e);
  }
  return RX_OK;
}

extern "C" rx_status rx_events_destroy(int32_t n, const rx_event_t* ev) {
  if (n < 0 || (n && !ev)) return rx_internal::set_error(RX_ERR_INVALID, "rx_events_destroy");
  for (int32_t i = 0; i < n; ++i)
    if (ev[i]) cudaEventDestroy(reinterpret_cast<cudaEvent_t>(ev[i]));
  return RX_OK;
}

extern "C" rx_status rx_event_elapsed_ms(rx_event_t start, rx_event_t end, float* out_ms) {
  if (!start || !end || !out_ms)
    return rx_internal::set_error(RX_ERR_INVALID, "rx_event_elapsed_ms: bad argument");
  if (cudaEventElapsedTime(out_ms, reinterpret_cast<cudaEvent_t>(start),
                           reinterpret_cast<cudaEvent_t>(end)) != cudaSuccess)
    return rx_internal::launch_status("rx_event_elapsed_ms");
  return RX_OK;
}
