// S6-S9: the C entry points of extend and decode attention over the radix KV
// pool, the log-sum-exp merge of decode partials, and the head_dim 256 decode
// tile kernel on warp-level tensor cores (mma.sync m16n8k16 bf16, fp32
// accumulate).  Extend attention and head_dim 128 decode run on the tcgen05
// kernels of attention_tc.cu.
//
// What is computed ("SGLang: Structured LLM Programs for Efficient
// Inference", sections "A quick recap of how an LLM generates text" and "How
// RadixAttention reuses past work"): each query attends, with softmax, over
// the keys of its request up to and including itself; keys of a reused prefix
// are read from the pool slots the radix cache handed out, exactly as if they
// had just been computed.  Query head h reads KV head h / (Hq/Hkv).
//
// In the mma.sync tile kernel one CTA owns a tile of query rows that all read
// the same KV head over the same key range, so every K/V tile staged in
// shared memory serves all of them:
//   extend: rows = (query token, head in group) of one request, token-major;
//           causal limit per row = prefix + token + 1;
//   decode: rows = (member request, head in group) of one plan work item: a
//           key chunk of a tree segment shared by the members (a dense
//           multi-query tile) or a request's private tail.  The CTA writes a
//           partial (o, lse) per row; a merge kernel combines the partials of
//           each request by log-sum-exp.
// K/V rows are gathered by slot with 16-byte cp.async into XOR-swizzled
// shared memory (double-buffered); QK^T and PV run on the tensor cores
// (ldmatrix + mma.sync); the softmax runs in registers with quad shuffles and
// exp2 on the SFU.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "ptx_util.cuh"
#include "rx.h"
#include "rx_internal.h"

// Bit 0: a slot read from req_to_token was outside [0, num_slots); slot 0 was
// used instead.  Read by rx_device_check().
static __device__ int32_t g_attention_error;

namespace {

using bf16 = __nv_bfloat16;
constexpr int BN = rx_internal::kKeyTile;  // keys per tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct TileArgs {
  const bf16* q;
  const bf16* kpool;  // layer base, [Hkv][num_slots][D]
  const bf16* vpool;
  int64_t head_stride;  // num_slots * D elements
  int64_t num_slots;
  const int32_t* table;
  int64_t row_stride;
  int hq;
  int group;
  float scale_log2;  // scale * log2(e)
  // extend
  const int32_t* req_rows;
  const int32_t* prefix_len;
  const int32_t* qo_indptr;
  const int32_t* tile_indptr;
  int num_req;
  int num_tiles;
  float* out;
  float* lse;
  // decode
  const int32_t* work;
  const int32_t* members;
  float* ws_o;
  float* ws_lse;
  int step;  // step index within a multi-step decode plan
};

// Shared-memory byte address of 16-byte chunk `chunk` of row `row` in a tile
// of D-wide bf16 rows; chunks are XOR-swizzled by the row's low 3 bits so
// ldmatrix row groups hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + uint32_t(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

struct Tile {
  const int32_t* trow;  // req_to_token row of the key source
  int key_begin, key_end;
  int nomask_end;  // keys below this are visible to every row of the tile
  int n_rows;
  // extend
  int gr0, q_base, prefix;
  // decode
  int member_off, part_base;
};

template <int BM, bool DECODE>
__device__ __forceinline__ Tile describe_tile(const TileArgs& a) {
  Tile t;
  if constexpr (DECODE) {
    const int32_t* w = a.work + int64_t(blockIdx.x) * RX_WORK_WORDS;
    t.trow = a.table + int64_t(w[0]) * a.row_stride;
    t.key_begin = w[1];
    t.key_end = w[7] > 0 ? min(w[2], w[7] + a.step) : w[2];  // growing private tail
    t.member_off = w[3];
    t.part_base = w[5];
    t.n_rows = w[6];
    t.nomask_end = t.key_end;
    t.gr0 = t.q_base = t.prefix = 0;
  } else {
    // heaviest tiles (last query tokens of a request) first
    const int tile = a.num_tiles - 1 - int(blockIdx.x);
    int lo = 0, hi = a.num_req;  // largest r with tile_indptr[r] <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.tile_indptr[mid] <= tile) lo = mid; else hi = mid;
    }
    const int G = a.group;
    t.q_base = a.qo_indptr[lo];
    const int s_r = a.qo_indptr[lo + 1] - t.q_base;
    t.prefix = a.prefix_len[lo];
    t.trow = a.table + int64_t(a.req_rows[lo]) * a.row_stride;
    t.gr0 = (tile - a.tile_indptr[lo]) * BM;
    t.n_rows = min(BM, s_r * G - t.gr0);
    const int t_first = t.gr0 / G;
    const int t_last = (t.gr0 + t.n_rows - 1) / G;
    t.key_begin = 0;
    t.key_end = t.prefix + t_last + 1;
    t.nomask_end = t.prefix + t_first + 1;
    t.member_off = t.part_base = 0;
  }
  return t;
}

// Query row i of the tile -> (query index, head, causal key limit).
template <bool DECODE>
__device__ __forceinline__ void row_of(const TileArgs& a, const Tile& t, int kvh, int i,
                                       int64_t& qi, int& head, int& lim) {
  const int G = a.group;
  if constexpr (DECODE) {
    const int unit = i / G;
    qi = a.members[t.member_off + unit];
    head = kvh * G + (i - unit * G);
    lim = t.key_end;
  } else {
    const int gr = t.gr0 + i;
    const int tok = gr / G;
    qi = int64_t(t.q_base) + tok;
    head = kvh * G + (gr - tok * G);
    lim = t.prefix + tok + 1;
  }
}

template <int D, int NT>
__device__ __forceinline__ void load_kv_tile(const TileArgs& a, const Tile& t, int kvh, int k0,
                                             uint32_t sk, uint32_t sv, int tid) {
  constexpr int CPR = D / 8;
  const bf16* kb = a.kpool + int64_t(kvh) * a.head_stride;
  const bf16* vb = a.vpool + int64_t(kvh) * a.head_stride;
#pragma unroll 4
  for (int c = tid; c < BN * CPR; c += NT) {
    const int j = c / CPR;
    const int ch = c - j * CPR;
    const int key = k0 + j;
    const bool ok = key < t.key_end;
    int64_t slot = 0;
    if (ok) {
      slot = __ldg(t.trow + key);
      if (slot < 0 || slot >= a.num_slots) {
        atomicOr(&g_attention_error, 1);
        slot = 0;
      }
    }
    const int64_t off = slot * D + ch * 8;
    rxk::cp_async_16(swz<D>(sk, j, ch), kb + off, ok);
    rxk::cp_async_16(swz<D>(sv, j, ch), vb + off, ok);
  }
}

template <int D, int NW, bool DECODE>
__global__ void __launch_bounds__(NW * 32, 1) attn_tile_kernel(const TileArgs a) {
  constexpr int BM = NW * 16;
  constexpr int NT = NW * 32;
  constexpr int CPR = D / 8;
  constexpr int NDT = D / 8;   // 8-wide output column tiles per warp row block
  constexpr int NST = BN / 8;  // 8-wide score tiles
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = rxk::smem_addr(smem);
  const uint32_t sK = sQ + BM * D * 2;
  const uint32_t sV = sK + 2 * BN * D * 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kvh = blockIdx.y;
  const Tile t = describe_tile<BM, DECODE>(a);

  // Q tile -> shared memory (rows past n_rows are zero)
  for (int c = tid; c < BM * CPR; c += NT) {
    const int i = c / CPR;
    const int ch = c - i * CPR;
    const bool ok = i < t.n_rows;
    const bf16* src = a.q;
    if (ok) {
      int64_t qi;
      int head, lim;
      row_of<DECODE>(a, t, kvh, i, qi, head, lim);
      src = a.q + (qi * a.hq + head) * D + ch * 8;
    }
    rxk::cp_async_16(swz<D>(sQ, i, ch), src, ok);
  }
  const int n_tiles = (t.key_end - t.key_begin + BN - 1) / BN;
  if (n_tiles > 0) load_kv_tile<D, NT>(a, t, kvh, t.key_begin, sK, sV, tid);
  rxk::cp_async_commit();

  // this thread's two rows
  int lim[2];
  bool ok_row[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = warp * 16 + (lane >> 2) + e * 8;
    ok_row[e] = i < t.n_rows;
    int64_t qi;
    int head;
    if (ok_row[e]) row_of<DECODE>(a, t, kvh, i, qi, head, lim[e]);
    else lim[e] = t.key_end;
  }

  float o[NDT][4];
#pragma unroll
  for (int j = 0; j < NDT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int it = 0; it < n_tiles; ++it) {
    const int k0 = t.key_begin + it * BN;
    const int buf = it & 1;
    if (it + 1 < n_tiles) {
      load_kv_tile<D, NT>(a, t, kvh, k0 + BN, sK + (buf ^ 1) * BN * D * 2,
                          sV + (buf ^ 1) * BN * D * 2, tid);
      rxk::cp_async_commit();
      rxk::cp_async_wait<1>();
    } else {
      rxk::cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kb = sK + buf * BN * D * 2;
    const uint32_t vb = sV + buf * BN * D * 2;

    // S = Q K^T for this warp's 16 rows x BN keys
    float s[NST][4];
#pragma unroll
    for (int j = 0; j < NST; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      rxk::ldsm_x4(swz<D>(sQ, warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int jn = 0; jn < NST / 2; ++jn) {
        uint32_t b0, b1, b2, b3;
        const int key = jn * 16 + (lane & 7) + ((lane >> 4) << 3);
        rxk::ldsm_x4(swz<D>(kb, key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        rxk::mma_bf16(s[2 * jn], a0, a1, a2, a3, b0, b1);
        rxk::mma_bf16(s[2 * jn + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // scale, mask, online softmax (log2 domain)
    const bool need_mask = k0 + BN > t.nomask_end;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NST; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[j][e] * a.scale_log2;
        if (need_mask) {
          const int key = k0 + j * 8 + 2 * (lane & 3) + (e & 1);
          if (key >= lim[e >> 1]) v = -INFINITY;
        }
        s[j][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float alpha[2], m_use[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 1));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 2));
      const float m_new = fmaxf(m_run[e], mx[e]);
      m_use[e] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[e] = rxk::fast_exp2(m_run[e] - m_use[e]);
      m_run[e] = m_new;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NST; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = rxk::fast_exp2(s[j][e] - m_use[e >> 1]);
        s[j][e] = p;
        rs[e >> 1] += p;
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) l_run[e] = l_run[e] * alpha[e] + rs[e];
#pragma unroll
    for (int j = 0; j < NDT; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      const uint32_t a0 = rxk::pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t a1 = rxk::pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t a2 = rxk::pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t a3 = rxk::pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int dn = 0; dn < NDT / 2; ++dn) {
        uint32_t b0, b1, b2, b3;
        rxk::ldsm_x4_t(swz<D>(vb, key, dn * 2 + (lane >> 4)), b0, b1, b2, b3);
        rxk::mma_bf16(o[2 * dn], a0, a1, a2, a3, b0, b1);
        rxk::mma_bf16(o[2 * dn + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // buffer `buf` is refilled two iterations later
  }

  // normalise and write
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float l = l_run[e];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int i = warp * 16 + (lane >> 2) + e * 8;
    if (!ok_row[e]) continue;
    int64_t qi;
    int head, lim_unused;
    row_of<DECODE>(a, t, kvh, i, qi, head, lim_unused);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = (m_run[e] == -INFINITY) ? -INFINITY : m_run[e] * kLn2 + logf(l);
    float* dst;
    float* lse_dst;
    if constexpr (DECODE) {
      const int unit = i / a.group;
      const int64_t part = int64_t(t.part_base) + unit;
      dst = a.ws_o + (part * a.hq + head) * D;
      lse_dst = a.ws_lse + part * a.hq + head;
    } else {
      dst = a.out + (qi * a.hq + head) * D;
      lse_dst = a.lse + qi * a.hq + head;
    }
#pragma unroll
    for (int j = 0; j < NDT; ++j) {
      const int col = j * 8 + 2 * (lane & 3);
      *reinterpret_cast<float2*>(dst + col) = make_float2(o[j][2 * e] * inv, o[j][2 * e + 1] * inv);
    }
    if ((lane & 3) == 0) *lse_dst = lse;
  }
}

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
                                                        int32_t* __restrict__ counter) {
  constexpr int V = D / 128;  // float4 per lane
  constexpr int CH = 8;       // part rows loaded together
  // launched after the decode kernel with programmatic stream serialization:
  // let the next step's kernel start launching, then wait for the partials
  rxk::griddep_launch_dependents();
  const int gw = int(blockIdx.x) * 8 + int(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const bool active = gw < B * hq;
  const int b = active ? gw / hq : 0;
  const int h = active ? gw - b * hq : 0;
  const int p0 = active ? indptr[b] : 0;
  const int n = active ? indptr[b + 1] - p0 : 0;
  int64_t e = lane < n ? int64_t(parts[p0 + lane]) * hq + h : 0;
  rxk::griddep_wait();
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

template <int D, int NW, bool DECODE>
constexpr int smem_bytes() {
  return (NW * 16 * D + 4 * BN * D) * 2;
}

template <int D, int NW, bool DECODE>
rx_status launch_tiles(const TileArgs& a, unsigned gx, unsigned gy, cudaStream_t s) {
  constexpr int bytes = smem_bytes<D, NW, DECODE>();
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(attn_tile_kernel<D, NW, DECODE>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    configured = true;
  }
  attn_tile_kernel<D, NW, DECODE><<<dim3(gx, gy), NW * 32, bytes, s>>>(a);
  return rx_internal::launch_status(DECODE ? "decode attention" : "extend attention");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace rx_internal {
int32_t attention_error_flags(bool clear) {
  int32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_attention_error, sizeof(v));
  if (clear && v) {
    int32_t z = 0;
    cudaMemcpyToSymbol(g_attention_error, &z, sizeof(z));
  }
  return v;
}
}  // namespace rx_internal

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
  if (R < 0 || num_tiles < 0 || num_tiles > INT32_MAX)
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
                                const int32_t* slots_new = nullptr) {
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
  TileArgs a{};
  a.q = static_cast<const bf16*>(d_q);
  const int64_t layer_off = int64_t(layer) * pool->num_kv_heads * pool->num_slots * D;
  a.kpool = static_cast<const bf16*>(pool->k_pool) + layer_off;
  a.vpool = static_cast<const bf16*>(pool->v_pool) + layer_off;
  a.head_stride = pool->num_slots * D;
  a.num_slots = pool->num_slots;
  a.table = d_req_to_token;
  a.row_stride = row_stride;
  a.hq = num_q_heads;
  a.group = num_q_heads / pool->num_kv_heads;
  a.scale_log2 = scale * kLog2e;
  a.work = d_plan + info->off_work;
  a.members = d_plan + info->off_members;
  a.step = step;
  const int64_t o_bytes = info->n_parts * num_q_heads * int64_t(D) * 4;
  a.ws_o = static_cast<float*>(d_workspace);
  a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(d_workspace) + ((o_bytes + 255) / 256) * 256);
  const int64_t l_bytes = info->n_parts * num_q_heads * 4;
  int32_t* counter = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(a.ws_lse) +
                                                ((l_bytes + 255) / 256) * 256);
  // the work counter of the decode kernel is 0 at every launch: zeroed here
  // once per call, reset by each merge after that
  if (D == 128 && first_call && cudaMemsetAsync(counter, 0, sizeof(int32_t), s) != cudaSuccess)
    return rx_internal::launch_status("decode counter reset");
  if (info->n_work > 0) {
    const int64_t n_small = info->n_work - info->n_work_tc;
    if (D == 128) {
      st = rx_internal::decode_fused(pool, layer, d_q, num_q_heads, d_req_to_token, row_stride,
                                     a.work, n_small, a.work + n_small * RX_WORK_WORDS,
                                     info->n_work_tc, a.members, scale, a.ws_o, a.ws_lse,
                                     counter, step, k_new, v_new, slots_new, s);
      if (st != RX_OK) return st;
    } else {
      st = launch_tiles<256, 4, true>(a, unsigned(info->n_work), pool->num_kv_heads, s);
      if (st != RX_OK) return st;
    }
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
  const float* wo = a.ws_o;
  const float* wl = a.ws_lse;
  if (D == 128)
    cudaLaunchKernelEx(&cfg, lse_merge_kernel<128>, indptr, parts, wo, wl, int(num_q_heads),
                       int(B), d_out, d_lse, counter);
  else
    cudaLaunchKernelEx(&cfg, lse_merge_kernel<256>, indptr, parts, wo, wl, int(num_q_heads),
                       int(B), d_out, d_lse, static_cast<int32_t*>(nullptr));
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
  for (int32_t i = 0; i < n_steps; ++i) {
    const rx_decode_step& st = steps[i];
    // every step's new token is the end of a growing private tail: the warp
    // kernel stores it itself
    const bool fused = B > 0 && pool->head_dim == 128 && G <= rx_internal::kDecodeSmallRows &&
                       st.info && st.info->tails_private == 1;
    if (!fused) {
      r = rx_kv_store(pool, layer, st.d_slots, st.d_k, st.d_v, B, stream);
      if (r != RX_OK) return r;
    } else if (!st.d_k || !st.d_v || !st.d_slots || (reinterpret_cast<uintptr_t>(st.d_k) & 15) ||
               (reinterpret_cast<uintptr_t>(st.d_v) & 15)) {
      return rx_internal::set_error(RX_ERR_INVALID, "rx_decode_steps: NULL or misaligned K/V");
    }
    r = decode_attention_impl(pool, layer, st.d_q, num_q_heads, d_req_to_token, row_stride,
                              st.d_plan, st.info, B, scale, st.d_out, st.d_lse, d_workspace,
                              workspace_bytes, reinterpret_cast<cudaStream_t>(stream), i == 0,
                              st.step, fused ? st.d_k : nullptr, fused ? st.d_v : nullptr,
                              fused ? st.d_slots : nullptr);
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
