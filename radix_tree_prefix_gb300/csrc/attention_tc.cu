// S6-S8: extend and decode attention on the 5th-generation tensor cores
// (tcgen05, TMEM), plus the warp role that decode adds for work items of few
// query rows; decode runs both in one launch per step (decode_fused_kernel).
//
// What is computed ("SGLang: Structured LLM Programs for Efficient
// Inference", sections "A quick recap of how an LLM generates text" and "How
// RadixAttention reuses past work"): every suffix query attends with softmax
// over its request's keys up to and including itself; reused prefix keys are
// read from the slots the radix cache handed out, as if just computed.
//
// One tile = 128 query rows that read one KV head over one key range:
//   extend: rows = (suffix token, head in group) of one request, token-major,
//           causal limit per row = prefix + token + 1;
//   decode: rows = (member request, head in group) of a tree segment chunk
//           shared by the members; writes partial (o, lse) per row.
// The tile (tc_tile3, 384 threads) streams K and V tiles of 32 KB (128 keys
// at head_dim 128, 64 at head_dim 256):
//   warps 0-7  softmax in two warpgroups that split every key tile's keys;
//              thread (w, i) owns query row i = TMEM lane i; the two halves
//              of a row agree on its max through shared memory; P (bf16)
//              goes into TMEM over the S tile it came from; O is rescaled in
//              TMEM when the max grows by more than 2^8 (rare after the
//              first tile); then the output is written;
//   warp 8     allocates TMEM and issues S_j = Q K_j^T (tcgen05.mma from
//              one thread) into a ring of three TMEM buffers, ahead of the
//              softmax;
//   warp 11    issues O += P_j V_j with P_j read from TMEM (O stays in TMEM
//              for the whole key loop);
//   warps 9-10 load K and V into 128-byte swizzled shared memory (three and
//              two stages): a tile whose slots form one contiguous run (the
//              allocator hands out runs, so this is the common case) is one
//              TMA box load per 64 columns; any other tile, and the ragged
//              last tile, is gathered slot by slot with 16-byte cp.async
//              (rows past the key range are zero-filled).
// Every mbarrier wait is bounded (about 2 s); on a timeout the CTA sets an
// error bit, drains its tensor-core work and frees TMEM before returning.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>

#include "ptx_util.cuh"
#include "rx.h"
#include "rx_internal.h"
#include "tc_util.cuh"

// Bit 0: a slot outside [0, num_slots) was read (slot 0 used instead);
// bit 1: a barrier wait timed out; bit 2: a tile found its dynamic shared
// memory off a 1024-byte boundary and did nothing.  Read by rx_device_check().
static __device__ int32_t g_tc_error;


namespace {

using bf16 = __nv_bfloat16;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (~2 s)
constexpr float kRescaleThreshold = 8.0f;       // log2 units
constexpr uint32_t kSleepNs = 0;                // MMA / loader waits: plain try_wait polling
constexpr float kMasked = -1.0e30f;             // raw score of a masked key
constexpr int kExtendInterleaveWaves = 8;
// Extend CTA order: heads interleaved also when one request's keys over all
// KV heads (K and V, bf16) take at most this much: the row tiles in flight
// then read a few requests' keys, which stay in L2 for every head at once.
constexpr int64_t kExtendInterleaveKvBytes = 32ll << 20;
constexpr int BM = 128;

struct TcArgs {
  const bf16* q;
  const bf16* kpool;  // layer base, [Hkv][num_slots][D]
  const bf16* vpool;
  int64_t head_stride;
  int64_t num_slots;
  const int32_t* table;
  int64_t row_stride;
  int hq;
  int group;
  float scale_log2;
  // extend
  const int32_t* req_rows;
  const int32_t* prefix_len;
  const int32_t* qo_indptr;
  const int32_t* tile_indptr;
  int num_req;
  int num_tiles;
  int heads_interleaved;   // extend CTA order: 1 = tile-major over heads, 0 = head-major
  float* out;
  float* lse;
  int64_t tma_row_base;  // row of (layer, KV head 0, slot 0) in the tensor maps
  int64_t tma_head_rows; // rows per KV head (num_slots)
  // decode
  const int32_t* work;     // tensor-core items
  const int32_t* members;
  float* ws_o;
  float* ws_lse;
  // fused decode: warp-role items (<= 16 rows) and the step's new tokens
  const int32_t* work_small;
  int n_small_units;       // warp-role (item, KV head) units
  int n_tc_ctas;           // tensor-core CTAs
  int n_warp_first;        // warp-role-only CTAs placed before them
  int* unit_counter;       // next warp-role unit to take (0 at launch)
  int tiles_leave;         // decode: tile CTAs exit after their tile
  int early_inputs;        // decode: the tiles may read Q and shared-segment keys
                           // before griddepcontrol.wait (see decode_fused)
  int step;                // step index within a multi-step plan
  const bf16* k_new;       // bf16 [B][Hkv][D] of the step's tokens, or NULL
  const bf16* v_new;
  const int32_t* slots_new;
};

struct TileDesc {
  const int32_t* trow;
  int key_begin, key_end, nomask_end, n_rows;
  int gr0, q_base, prefix;
  int member_off, part_base;
};

template <bool DECODE>
__device__ __forceinline__ TileDesc describe(const TcArgs& a, int bx) {
  TileDesc t;
  if constexpr (DECODE) {
    const int32_t* w = a.work + int64_t(bx) * RX_WORK_WORDS;
    t.trow = a.table + int64_t(w[0]) * a.row_stride;
    t.key_begin = w[1];
    t.key_end = w[2];
    t.member_off = w[3];
    t.part_base = w[5];
    t.n_rows = w[6];
    t.nomask_end = t.key_end;
    t.gr0 = t.q_base = t.prefix = 0;
  } else {
    const int tile = a.num_tiles - 1 - bx;  // heaviest first
    // the request of this tile: the last r with tile_indptr[r] <= tile, found
    // by the warp in rounds of 32 samples (each round one load per lane and
    // a ballot) instead of a binary search's chain of dependent loads, which
    // held every CTA's start-up for several microseconds
    const int ln = int(threadIdx.x & 31);
    int lo = 0, hi = a.num_req;
    while (hi - lo > 32) {
      const int step = (hi - lo + 31) >> 5;
      const int p = lo + ln * step;
      const bool le = p < hi && __ldg(a.tile_indptr + p) <= tile;
      const int k = 31 - __clz(__ballot_sync(0xffffffffu, le));  // lane 0's sample is <= tile
      lo = lo + k * step;
      hi = min(hi, lo + step);
    }
    {
      const int p = lo + ln;
      const bool le = p < hi && __ldg(a.tile_indptr + p) <= tile;
      lo += 31 - __clz(__ballot_sync(0xffffffffu, le));
    }
    const int G = a.group;
    t.q_base = a.qo_indptr[lo];
    const int s_r = a.qo_indptr[lo + 1] - t.q_base;
    t.prefix = a.prefix_len[lo];
    t.trow = a.table + int64_t(a.req_rows[lo]) * a.row_stride;
    t.gr0 = (tile - a.tile_indptr[lo]) * BM;
    t.n_rows = min(BM, s_r * G - t.gr0);
    t.key_begin = 0;
    t.key_end = t.prefix + (t.gr0 + t.n_rows - 1) / G + 1;
    t.nomask_end = t.prefix + t.gr0 / G + 1;
    t.member_off = t.part_base = 0;
  }
  return t;
}

// row i -> (query index, head, part index for decode, causal limit)
template <bool DECODE>
__device__ __forceinline__ void row_info(const TcArgs& a, const TileDesc& t, int kvh, int i,
                                         int64_t& qi, int& head, int64_t& part, int& lim) {
  const int G = a.group;
  if constexpr (DECODE) {
    const int unit = i / G;
    qi = a.members[t.member_off + unit];
    head = kvh * G + (i - unit * G);
    part = int64_t(t.part_base) + unit;
    lim = t.key_end;
  } else {
    const int gr = t.gr0 + i;
    const int tok = gr / G;
    qi = int64_t(t.q_base) + tok;
    head = kvh * G + (gr - tok * G);
    part = 0;
    lim = t.prefix + tok + 1;
  }
}

// 128-byte-swizzled tile of `rows` rows, stored as column blocks of 64 bf16:
// byte address of 16-byte chunk `ch` (of the full row) of row r.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int rows, int r, int ch) {
  return base + uint32_t((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// Tensor-core tile: 128 query rows, key tiles of BN = 128 keys at head_dim
// 128 and 64 at head_dim 256 (a K or V tile is 32 KB either way), 384
// threads.  The MMA warps keep S tiles ahead of the softmax: S_{j+2} =
// Q K_{j+2}^T is issued before PV_j, into a ring of three S buffers in TMEM,
// so the softmax of tile j+1 never waits for an MMA.  P_j (bf16, two keys per
// column) overwrites the first BN/2 columns of S_j's buffer once the softmax
// has read S_j, and PV_j reads it from TMEM as its A operand; the S issuer
// waits for PV_j's completion (barrier pf) before S_{j+3} reuses that
// buffer.
// TMEM: S ring [0, 3 BN), O from column O_COL (D columns).  Shared memory: Q
// (128-byte swizzled, the A operand of S), K in three stages, V in two.
// Warps 0-7 softmax in two warpgroups that split each key tile's columns
// (thread (w, i) of warpgroup w: row i = TMEM lane i, keys [w BN/2, (w+1)
// BN/2); it also gathers half of Q row i first), warp 8 issues the S MMAs
// and warp 11 the PV MMAs (two instruction streams: one thread issuing all
// of a key tile's MMAs set the tile's period), warp 9 loads K and warp 10
// loads V (a V stage frees only when PV of its previous tile completes, and
// K loads must not queue behind that).
// 12 warps: 0-7 softmax (two warpgroups), 8 S = Q K^T issue, 9 K loader, 10 V
// loader, 11 O += P V issue
constexpr int kThreads3 = 384;

template <int HEAD_DIM>
struct Layout3 {
  static constexpr int D = HEAD_DIM;
  static constexpr int BN = D == 128 ? 128 : 64;
  static constexpr int KSTAGES = 3, VSTAGES = 2, SBUF = 3;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int Q = 0;
  static constexpr int K0 = Q + BM * D * 2;
  static constexpr int V0 = K0 + KSTAGES * KV_BYTES;
  // exchange slots: per-tile half-row maxima, two parities, [2][2
  // warpgroups][128 rows] floats; the final row sums reuse the parity that
  // follows the last tile
  static constexpr int XCH = V0 + VSTAGES * KV_BYTES;
  static constexpr int BAR = XCH + 2 * 2 * 128 * 4;
  // barriers: q, kfull, vfull (one per stage), s[3], p[3], o[2] (PV of even
  // / odd tiles), final, max exchange[2], sum exchange, pf[3] (PV of the P
  // in S buffer b done, so S may overwrite it).  A K stage is free
  // again when the S product that read it completes (s[] of the same index:
  // both rings have three entries) and a V stage when its PV product does
  // (o[] of the same parity: two V stages).
  static constexpr int NBAR = 1 + KSTAGES + VSTAGES + 2 * SBUF + 6 + SBUF;
  static_assert(KSTAGES == SBUF && VSTAGES == 2, "stage rings share the MMA barriers");
  static constexpr int MISC = BAR + NBAR * 8;  // tmem address, abort flag
  // At head_dim 128 the layout carries 1024 bytes of slack to align the
  // swizzled tiles.  At head_dim 256 it leaves under 1 KB of the 227 KB a CTA
  // may have, so the tile requires dynamic shared memory that starts on a
  // 1024-byte boundary: a CTA that finds otherwise sets an error bit and
  // returns without touching anything.
  static constexpr bool SLACK = D == 128;
  static constexpr int BYTES = MISC + 16 + (SLACK ? 1024 : 0);
  static constexpr int TMEM_COLS = 512;
  static constexpr int O_COL = D == 128 ? SBUF * BN : 256;
  static_assert(SBUF * BN <= O_COL && O_COL + D <= TMEM_COLS, "TMEM budget");
  static_assert(BYTES <= 227 * 1024, "shared memory budget");
};

// D(tmem) (+)= A * B(smem), A from shared memory (ss) or TMEM (ts), issued
// by a single thread, with the shared-memory descriptors passed as 32-bit
// halves: the high half (stride between 8-row groups, version, swizzle) is
// common to every operand of the tile, and the low half (start address >> 4
// and leading-byte offset) moves by compile-time steps, so the issuing thread
// spends one add per operand instead of rebuilding 64-bit descriptors.
__device__ __forceinline__ void mma_ss_split(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 ad, bd;\n setp.ne.b32 p, %5, 0;\n"
      " mov.b64 ad, {%1, %3};\n mov.b64 bd, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_split(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 bd;\n setp.ne.b32 p, %5, 0;\n"
      " mov.b64 bd, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns of 32-bit values from registers (thread t: lane t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

template <int D, bool DECODE>
__device__ __forceinline__ void tc_tile3(const TcArgs& a, const CUtensorMap* tmk,
                                         const CUtensorMap* tmv, uint8_t* smem_raw, int bx,
                                         int kvh) {
  using Lo = Layout3<D>;
  constexpr int BN = Lo::BN, NK = Lo::KSTAGES, NV = Lo::VSTAGES, NB = Lo::SBUF;
  const uint32_t raw = rxk::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte alignment of the swizzled tiles
  if constexpr (!Lo::SLACK) {
    if (base != raw) {  // uniform over the CTA: nothing initialised yet
      if (threadIdx.x == 0) atomicOr(&g_tc_error, 4);
      return;
    }
  }
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + Lo::Q;
  const uint32_t bar = base + Lo::BAR;
  const uint32_t BAR_Q = bar;
  // barrier indices: q, kfull[NK], vfull[NV], s[NB], p[NB], o[2], final,
  // max exchange[2], sum exchange
  auto BAR_KF = [&](int s) { return bar + 8u * (1 + s); };
  auto BAR_VF = [&](int s) { return bar + 8u * (1 + NK + s); };
  auto BAR_S = [&](int b) { return bar + 8u * (1 + NK + NV + b); };
  auto BAR_P = [&](int b) { return bar + 8u * (1 + NK + NV + NB + b); };
  constexpr uint32_t kAfterP = 1 + NK + NV + 2 * NB;
  // PV_j completes phase j / 2 of BAR_O(j % 2).  One barrier per parity of
  // j: when the softmax of tile j waits for PV_{j-1}, PV_{j-3} has completed
  // (it was issued before S_j, whose completion the softmax waited for), so the
  // phase parity it waits on cannot be mistaken for an older phase; with a
  // single barrier PV_{j-2} may still be in flight and the parity would be
  // ambiguous.
  auto BAR_O = [&](int p) { return bar + 8u * (kAfterP + p); };
  const uint32_t BAR_FIN = bar + 8u * (kAfterP + 2);
  auto XB = [&](int p) { return bar + 8u * (kAfterP + 3 + p); };
  const uint32_t XE = bar + 8u * (kAfterP + 5);
  // PV_j completes phase j / NB of BAR_PF(j % NB): S buffer j % NB is free
  // for S_{j+NB}
  auto BAR_PF = [&](int b) { return bar + 8u * (kAfterP + 6 + b); };
  static_assert(kAfterP + 6 + NB == Lo::NBAR, "barrier count");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Lo::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Lo::MISC + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const TileDesc t = describe<DECODE>(a, bx);
  const int n_tiles = (t.key_end - t.key_begin + BN - 1) / BN;

  // Softmax threads: the query row of their TMEM lane, and the gather of
  // half of Q row i, issued before the barriers and TMEM are set up so the
  // copies overlap that start-up (nothing else uses the Q buffer yet; the
  // arrival on the Q barrier follows the CTA-wide sync below).
  const int wg = warp >> 2;
  const int i = (warp & 3) * 32 + lane;  // TMEM lane
  // the tile row in lane i: row i, or with M = 64 products (at most 64
  // rows) row 16 (i / 32) + i % 16 in the first 16 lanes of each quadrant
  const bool m64 = t.n_rows <= 64;
  const int row = m64 ? (((i >> 5) << 4) | (i & 15)) : i;
  int64_t qi = 0, part = 0;
  int head = 0, lim = t.key_end;
  bool valid = false;
  if (warp < 8) {
    valid = (!m64 || (i & 16) == 0) && row < t.n_rows;
    if (valid) row_info<DECODE>(a, t, kvh, row, qi, head, part, lim);
    // the Q row this thread gathers: tile row i into shared-memory row i
    // (the A operand's rows, whatever the TMEM layout of the products)
    int64_t gqi = qi;
    int ghead = head;
    bool gvalid = valid;
    if (m64) {
      int64_t gpart = 0;
      int glim = 0;
      gqi = 0;
      ghead = 0;
      gvalid = i < t.n_rows;
      if (gvalid) row_info<DECODE>(a, t, kvh, i, gqi, ghead, gpart, glim);
    }
    // the queries (and, below, the outputs: decode's partial buffers the
    // previous merge read) are touched only once earlier kernels on the
    // stream are done; with early inputs the queries are complete already
    // and only the partial writes wait
    if (!DECODE || !a.early_inputs) rxk::griddep_wait();
    // chunks [8 w, 8 w + 8) of Q row i (zeros past the tile's rows) while
    // the loader warps already stream the first K/V tiles
    const bf16* src = a.q + (gqi * a.hq + ghead) * D;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const int ch = wg * (D / 16) + c;
      rxk::cp_async_16(sw128(sQ, BM, i, ch), src + ch * 8, gvalid);
    }
    rxk::cp_async_commit();
  }

  if (tid == 0) {
    tc::mbar_init(BAR_Q, 8 * 32);  // every softmax thread lands half a Q row
    for (int s = 0; s < NK; ++s) tc::mbar_init(BAR_KF(s), 1);
    for (int s = 0; s < NV; ++s) tc::mbar_init(BAR_VF(s), 1);
    for (int b = 0; b < NB; ++b) {
      tc::mbar_init(BAR_S(b), 1);
      tc::mbar_init(BAR_P(b), 8 * 32);
    }
    tc::mbar_init(XB(0), 8 * 32);
    tc::mbar_init(XB(1), 8 * 32);
    tc::mbar_init(XE, 8 * 32);
    tc::mbar_init(BAR_O(0), 1);
    tc::mbar_init(BAR_O(1), 1);
    tc::mbar_init(BAR_FIN, 2);  // one commit per issuing thread
    for (int b = 0; b < NB; ++b) tc::mbar_init(BAR_PF(b), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(rxk::smem_addr(tmem_slot), Lo::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------- loaders
    const bool load_v = warp == 10;
    // keys written by earlier kernels on the stream are read from here on
    // (a decode step after the first of a run reads shared segments that no
    // kernel of the run writes: it need not wait)
    if (!DECODE || !a.early_inputs) rxk::griddep_wait();
    constexpr int CPR = D / 8;
    constexpr int SPL = BN / 32;  // slots per lane: rows lane + 32 i
    const bf16* kb = a.kpool + int64_t(kvh) * a.head_stride;
    const bf16* vb = a.vpool + int64_t(kvh) * a.head_stride;
    const int64_t row0 = a.tma_row_base + int64_t(kvh) * a.tma_head_rows;
    // slots of four consecutive tiles (tile j in ring j % 4): a tile's table
    // reads are issued four tiles ahead into registers that nothing touches
    // until then, so their round trips to L2 overlap the loads before them
    int32_t sa[SPL], sb[SPL], sc[SPL], sd[SPL];
    auto load_slots = [&](int j, int32_t (&dst)[SPL]) {
      const int k0 = t.key_begin + j * BN;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const int key = k0 + lane + 32 * i;
        dst[i] = (j < n_tiles && key < t.key_end) ? __ldg(t.trow + key) : -1;
      }
    };
    auto check_slots = [&](int32_t (&slot)[SPL]) {
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        if (slot[i] >= a.num_slots || slot[i] < -1) {
          atomicOr(&g_tc_error, 1);
          slot[i] = 0;
        }
      }
    };
    // one K or V tile: TMA box loads if the slots are one contiguous run of
    // BN valid slots, else a zero-filling cp.async gather
    auto load_tile = [&](int32_t (&slot)[SPL], const CUtensorMap* tm, const bf16* src_base,
                         uint32_t dst, uint32_t full_bar) {
      const int32_t first = __shfl_sync(0xffffffffu, slot[0], 0);
      bool run = first >= 0 && int64_t(first) + BN <= a.num_slots;
#pragma unroll
      for (int i = 0; i < SPL; ++i) run = run && (slot[i] == first + lane + 32 * i);
      run = __all_sync(0xffffffffu, run);
      if (run) {
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(full_bar, uint32_t(BN * D * 2));
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            tc::tma_load_2d(dst + uint32_t(cb * BN * 128), tm, cb * 64, int(row0 + first),
                            full_bar);
        }
      } else {
        // lanes 0-15 and 16-31 copy chunks (lane % 16) + 16 h of rows 2k, 2k+1
#pragma unroll
        for (int i = 0; i < SPL; ++i) {
#pragma unroll 4
          for (int k = 0; k < 16; ++k) {
            const int row = 32 * i + 2 * k + (lane >> 4);
            const int32_t sl = __shfl_sync(0xffffffffu, slot[i], row & 31);
            const bool ok = sl >= 0;
            const int64_t s64 = ok ? int64_t(sl) : 0;
#pragma unroll
            for (int h = 0; h < CPR / 16; ++h) {
              const int ch = (lane & 15) + 16 * h;
              rxk::cp_async_16(sw128(dst, BN, row, ch), src_base + s64 * D + ch * 8, ok);
            }
          }
        }
        rxk::cp_async_commit();
        rxk::cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(full_bar);
      }
    };
    load_slots(0, sa);
    load_slots(1, sb);
    load_slots(2, sc);
    load_slots(3, sd);
    // tile j (K stage j % NK, V stage j % NV): K and V with the slots in
    // `slot`, then tile j + 4's table reads into the same registers; a stage
    // is refilled once the MMA that read its previous tile has completed:
    // S_{j-NK} (barrier s[j % NK]) for K, PV_{j-2} (barrier o[j % 2]) for V
    int issued = 0;  // tiles whose K (or V) load has been issued
    auto step = [&](int j, int32_t (&slot)[SPL]) -> bool {
      const int sk = j % NK, sv = j % NV;
      check_slots(slot);
      if (!load_v) {
        if (j >= NK &&
            !__all_sync(0xffffffffu, tc::mbar_wait(BAR_S(sk), uint32_t(j / NK - 1) & 1u,
                                                    abort_flag, kWaitLimit, kSleepNs)))
          return false;
        load_tile(slot, tmk, kb, base + Lo::K0 + sk * Lo::KV_BYTES, BAR_KF(sk));
      } else {
        if (j >= NV &&
            !__all_sync(0xffffffffu, tc::mbar_wait(BAR_O(sv), uint32_t(j / NV - 1) & 1u,
                                                    abort_flag, kWaitLimit, kSleepNs)))
          return false;
        load_tile(slot, tmv, vb, base + Lo::V0 + sv * Lo::KV_BYTES, BAR_VF(sv));
      }
      issued = j + 1;
      load_slots(j + 4, slot);
      return true;
    };
    for (int j = 0; j < n_tiles; j += 4) {
      if (!step(j, sa)) break;
      if (j + 1 < n_tiles && !step(j + 1, sb)) break;
      if (j + 2 < n_tiles && !step(j + 2, sc)) break;
      if (j + 3 < n_tiles && !step(j + 3, sd)) break;
    }
    // Before the CTA gives up its shared memory, the last load of every
    // stage has landed.  On the normal path the MMAs consumed them all and
    // these waits return at once; after a wait of another warp timed out
    // (abort), TMA box loads may still be in flight, so they get one more
    // bounded wait that does not look at the abort flag.
    if (lane == 0) {
      const int NS = load_v ? NV : NK;
      int drain_abort = 0;
      for (int j = issued > NS ? issued - NS : 0; j < issued; ++j) {
        const uint32_t fb = load_v ? BAR_VF(j % NV) : BAR_KF(j % NK);
        tc::mbar_wait(fb, uint32_t(j / NS) & 1u, &drain_abort, kWaitLimit);
      }
    }
    __syncwarp();
  } else if (warp == 8 || warp == 11) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads, so neither instruction stream alone sets the key
    // tile's period: warp 8 issues S_j = Q K_j^T into S buffer j % 3, warp 11
    // issues O += P_j V_j with P_j from TMEM.  The two streams no longer
    // complete in one order, so the S issuer waits, before S_j, until PV_{j-3}
    // (which read P_{j-3} from the same buffer) has completed (barrier pf[j %
    // 3]); hence S_j completing still implies PV_{j-3} completed, which the
    // softmax's wait on o[] relies on.
    if (lane == 0) {
      // a tile of at most 64 rows runs M = 64 products (half the MMA work;
      // its row r then sits in TMEM lane 32 (r / 16) + r % 16)
      const bool m64 = t.n_rows <= 64;
      const uint32_t IDESC_S = m64 ? tc::idesc_bf16(64, BN, 0) : tc::idesc_bf16(BM, BN, 0);
      const uint32_t IDESC_PV = m64 ? tc::idesc_bf16(64, D, 1) : tc::idesc_bf16(BM, D, 1);
      // shared-memory descriptors (128-byte swizzle, 1024 bytes between
      // 8-row groups): common high half; low halves of Q, K stage 0 (K-major,
      // leading offset 16 B) and V stage 0 (MN-major, leading offset = one
      // 64-column block of BN rows).  Fields of the 64-bit descriptor: start
      // address >> 4 in bits 0-13, leading byte offset >> 4 in bits 16-29,
      // stride byte offset >> 4 in bits 32-45, version 1 at bit 46, layout
      // (2 = 128-byte swizzle) in bits 61-63; swizzle atoms (8 rows x 128 B)
      // start on 1024-byte boundaries
      constexpr uint32_t DHI = (1024u >> 4) | (1u << 14) | (2u << 29);
      constexpr uint32_t KV_STEP = uint32_t(Lo::KV_BYTES) >> 4;
      static_assert(Lo::V0 + NV * Lo::KV_BYTES < (1 << 18), "descriptor address field");
      if (warp == 8) {
        const uint32_t q_lo = ((sQ & 0x3FFFFu) >> 4) | (1u << 16);
        const uint32_t k_lo0 = (((base + Lo::K0) & 0x3FFFFu) >> 4) | (1u << 16);
        const bool ok = tc::mbar_wait(BAR_Q, 0, abort_flag, kWaitLimit, kSleepNs);
        // S_j's K stage and S buffer (the same index: both rings have NB
        // entries) and the phases of its waits
        int sb = 0;
        uint32_t k_phase = 0, pf_phase = 0;
        for (int j = 0; ok && j < n_tiles; ++j) {
          if (j >= NB && !tc::mbar_wait(BAR_PF(sb), pf_phase, abort_flag, kWaitLimit, kSleepNs))
            break;
          if (!tc::mbar_wait(BAR_KF(sb), k_phase, abort_flag, kWaitLimit, kSleepNs)) break;
          tc::tc_fence_after();
          const uint32_t k_lo = k_lo0 + uint32_t(sb) * KV_STEP;
          const uint32_t d_s = tmem + uint32_t(sb * BN);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t a_off = uint32_t(((ks >> 2) * (BM * 128) + (ks & 3) * 32) >> 4);
            const uint32_t b_off = uint32_t(((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4);
            mma_ss_split(d_s, q_lo + a_off, k_lo + b_off, DHI, IDESC_S, ks > 0 ? 1u : 0u);
          }
          tc::mma_commit(BAR_S(sb));  // also frees K stage sb
          if (++sb == NB) {
            sb = 0;
            k_phase ^= 1u;
            if (j >= NB) pf_phase ^= 1u;
          }
        }
      } else {
        const uint32_t v_lo0 =
            (((base + Lo::V0) & 0x3FFFFu) >> 4) | (uint32_t(BN * 128 / 16) << 16);
        int sv = 0, pb = 0;
        uint32_t v_phase = 0, p_phase = 0;
        for (int j = 0; j < n_tiles; ++j) {
          if (!tc::mbar_wait(BAR_P(pb), p_phase, abort_flag, kWaitLimit, kSleepNs)) break;
          if (!tc::mbar_wait(BAR_VF(sv), v_phase, abort_flag, kWaitLimit, kSleepNs)) break;
          tc::tc_fence_after();
          const uint32_t v_lo = v_lo0 + uint32_t(sv) * KV_STEP;
          const uint32_t p_t = tmem + uint32_t(pb * BN);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            mma_ts_split(tmem + uint32_t(Lo::O_COL), p_t + uint32_t(ks * 8),
                         v_lo + uint32_t(ks * 2048 / 16), DHI, IDESC_PV,
                         (j > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(BAR_O(j & 1));  // also frees V stage sv (== j & 1)
          tc::mma_commit(BAR_PF(pb));    // S buffer pb may take S_{j+3}
          if (++sv == NV) {
            sv = 0;
            v_phase ^= 1u;
          }
          if (++pb == NB) {
            pb = 0;
            p_phase ^= 1u;
          }
        }
      }
      // drain: every MMA this thread issued has completed once the final
      // barrier (one arrival per issuing thread) completes.  The wait ignores
      // the abort flag (bounded all the same): after another warp gave up,
      // MMAs already issued must finish writing TMEM and reading shared
      // memory before the CTA frees both.
      tc::mma_commit(BAR_FIN);
      int drain_abort = 0;
      tc::mbar_wait(BAR_FIN, 0, &drain_abort, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Two warpgroups: warpgroup w (warps 4w .. 4w+3) owns keys [64 w, 64 w +
    // 64) of every key tile for the same 128 rows (warp 4w + q reaches TMEM
    // lanes 32 q ..).  Per tile the two halves of a row agree on the row max
    // through shared memory (one bounded mbarrier round), so both write P
    // against the same reference and share one O accumulator.
    constexpr int HALF = BN / 2;
    const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
    float* xch = reinterpret_cast<float*>(gbase + Lo::XCH);  // [2][2 warpgroups][BM]
    // the Q gather issued at the start has landed
    rxk::cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(BAR_Q);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % NB;  // S buffer
      // waits are made warp-uniform before any warp-collective tcgen05 op
      if (!__all_sync(0xffffffffu, tc::mbar_wait(BAR_S(s), uint32_t(j / NB) & 1u, abort_flag,
                                                  kWaitLimit))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const int k0 = t.key_begin + j * BN + wg * HALF;  // first key of this half
      const bool need_mask = k0 + HALF > t.nomask_end;
      uint32_t sr[HALF];
      tc::tmem_ld_row<HALF>(tl + uint32_t(s * BN + wg * HALF), sr);
      tc::tmem_ld_wait();
      // row max of the raw scores over this half (masked keys get a large
      // negative finite score, so no exponent below is an infinity or a NaN,
      // even for a row whose keys are all masked); eight independent partial
      // maxima keep the chains short
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = kMasked;
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < HALF; ++e) {
          if (k0 + e >= lim) sr[e] = __float_as_uint(kMasked);
          mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sr[e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < HALF; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sr[e]));
      }
      const float mx_half = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                  fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // the other half's max of this row (parity-double-buffered slot: a thread
      // reaches tile j + 2's write only after every thread has passed tile
      // j + 1's exchange, hence has read tile j's)
      xch[((j & 1) * 2 + wg) * BM + i] = mx_half;
      tc::mbar_arrive(XB(j & 1));
      if (!__all_sync(0xffffffffu, tc::mbar_wait(XB(j & 1), (j >> 1) & 1, abort_flag, kWaitLimit))) {
        ok = false;
        break;
      }
      const float mx_other = xch[((j & 1) * 2 + (1 - wg)) * BM + i];
      const float mx = a.scale_log2 * fmaxf(mx_half, mx_other);
      const float m_new = fmaxf(m_ref, mx);
      if (j == 0) {
        m_ref = m_new;
      } else {
        const bool need = m_new > m_ref + kRescaleThreshold;
        // both warps of a row quadrant see the same rows, so they agree
        if (__any_sync(0xffffffffu, need)) {
          // O is rescaled once PV_{j-1} has written it; each warpgroup takes
          // half of its columns
          if (!__all_sync(0xffffffffu, tc::mbar_wait(BAR_O((j - 1) & 1), ((j - 1) >> 1) & 1,
                                                      abort_flag, kWaitLimit))) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const float alpha = need ? rxk::fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t r[32];
            const uint32_t col = uint32_t(Lo::O_COL + wg * (D / 2) + cc * 32);
            tc::tmem_ld32(tl + col, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tc::tmem_st32(tl + col, r);
          }
          if (need) {
            l *= alpha;
            m_ref = m_new;
          }
        }
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float l8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) l8[u] = 0.f;
#pragma unroll
      for (int cc = 0; cc < HALF / 32; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          // p = 2^(scale*s - m) for two keys: exp2 in fp32 on the SFU, then
          // both rounded to nearest into one bf16x2 word (the precision P has
          // in the PV product).  With the lazy max the dominant keys'
          // exponents reach +8, where a bf16 exponent or a bf16 exp2 result
          // would cost up to 1% per weight on peaked rows.  The row sum adds
          // exactly the rounded values in fp32, in eight independent partial
          // sums.
          const float x0 = fmaf(__uint_as_float(sr[cc * 32 + e]), a.scale_log2, -m_use);
          const float x1 = fmaf(__uint_as_float(sr[cc * 32 + e + 1]), a.scale_log2, -m_use);
          const uint32_t h = rxk::pack_bf16(rxk::fast_exp2(x0), rxk::fast_exp2(x1));
          l8[(e >> 1) & 7] += __uint_as_float(h << 16) + __uint_as_float(h & 0xffff0000u);
          pk[e >> 1] = h;
        }
        // keys of this half, two per column, over the first BN/2 columns
        // of S_j's buffer (half w at columns w BN/4 ..)
        tmem_st16(tl + uint32_t(s * BN + wg * (HALF / 2) + 16 * cc), pk);
      }
      l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(BAR_P(s));
    }
    // The epilogue waits on BAR_FIN, which completes exactly once, after every
    // MMA of the CTA, then the halves add
    // their row sums through shared memory and warpgroup w writes output
    // columns [64 w, 64 w + 64).  Every softmax thread arrives on the
    // exchange barrier, so no waiter is left behind when a wait gave up.
    const bool fin = ok && n_tiles > 0 &&
                     __all_sync(0xffffffffu, tc::mbar_wait(BAR_FIN, 0, abort_flag, kWaitLimit));
    if (DECODE && a.early_inputs) rxk::griddep_wait();  // the previous merge read ws
    // (a thread got here after every thread passed the exchange of tile
    // n_tiles - 1, hence had read the slot of tile n_tiles - 2)
    if (fin) xch[((n_tiles & 1) * 2 + wg) * BM + i] = l;
    tc::mbar_arrive(XE);
    const bool xok = __all_sync(0xffffffffu, tc::mbar_wait(XE, 0, abort_flag, kWaitLimit));
    if (fin && xok) {
      tc::tc_fence_after();
      const float l_all = l + xch[((n_tiles & 1) * 2 + (1 - wg)) * BM + i];
      const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
      float* dst;
      float* lse_dst;
      if constexpr (DECODE) {
        dst = a.ws_o + (part * a.hq + head) * D;
        lse_dst = a.ws_lse + part * a.hq + head;
      } else {
        dst = a.out + (qi * a.hq + head) * D;
        lse_dst = a.lse + qi * a.hq + head;
      }
      // Warpgroup w owns output columns [w D/2, (w+1) D/2).  Its rows go
      // through shared memory (the K stages, idle once every MMA completed
      // and every load landed) so that each warp then writes the 32 rows of
      // its TMEM lane quadrant as whole contiguous row segments: one thread
      // per row would make every store instruction touch 32 rows.
      constexpr int HC = D / 2;           // columns per warpgroup
      constexpr int PITCH = HC * 4 + 16;  // staged row bytes (+16: conflict-free)
      constexpr int LPR = HC / 4;         // float4 per staged row
      static_assert(2 * BM * PITCH <= Lo::XCH - Lo::K0, "staging fits in the K/V stages");
      uint8_t* stage = gbase + Lo::K0 + wg * (BM * PITCH);
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        uint32_t r[32];
        tc::tmem_ld32(tl + uint32_t(Lo::O_COL + wg * HC + cc * 32), r);
        tc::tmem_ld_wait();
        float4* s4 = reinterpret_cast<float4*>(stage + i * PITCH + cc * 128);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          s4[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                              __uint_as_float(r[4 * e + 2]) * inv,
                              __uint_as_float(r[4 * e + 3]) * inv);
      }
      __syncwarp();
      const int qrow = (warp & 3) * 32;  // first row of this warp's quadrant
      const unsigned long long my_dst =
          valid ? reinterpret_cast<unsigned long long>(dst + wg * HC) : 0ull;
#pragma unroll 4
      for (int k = 0; k < LPR; ++k) {
        const int idx = k * 32 + lane;
        const int rr = idx / LPR, c4 = idx - rr * LPR;  // row within the quadrant, float4
        const unsigned long long rd = __shfl_sync(0xffffffffu, my_dst, rr);
        const float4 v = *reinterpret_cast<const float4*>(stage + (qrow + rr) * PITCH + c4 * 16);
        if (rd) reinterpret_cast<float4*>(rd)[c4] = v;
      }
      if (valid && wg == 0) *lse_dst = m_ref * kLn2 + logf(l_all);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(&g_tc_error, 2);
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Lo::TMEM_COLS);
  }
}

// Extend: one tile per CTA, heaviest row tile first.  With heads_interleaved
// (few waves of CTAs, or short contexts) CTA c takes row tile c / Hkv of KV
// head c % Hkv, so the heavy tiles of every head go out before the light
// ones and the last wave is short; otherwise CTA c takes head c / tiles, so
// the CTAs resident at one time read the keys of one head and those stay in
// L2.
template <int D>
__global__ void __launch_bounds__(kThreads3, 1)
    attn_tc3_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int c = int(blockIdx.x);
  if (a.heads_interleaved) {
    const int hkv = a.hq / a.group;
    tc_tile3<D, false>(a, &tmk, &tmv, smem_raw, c / hkv, c - (c / hkv) * hkv);
  } else {
    tc_tile3<D, false>(a, &tmk, &tmv, smem_raw, c % a.num_tiles, c / a.num_tiles);
  }
}

// ---------------------------------------------------------------------------
// Warp role of the fused decode kernel: work items of <= 16 query rows at
// head_dim 128, <= 8 at 256 (a request's private tail, or a shared segment
// chunk with few rows).  One warp owns one (item, KV head) unit and streams its keys
// in steps of 16.  With few query rows per item the products are computed transposed,
// keys in the M dimension of mma.sync m16n8k16 and query rows in N (8 or 16
// rows, NR n-tiles), so no MMA row is wasted on keys:
//   S^T (16 keys x 8 rows)  = K (16 x D, ldmatrix)        . Q^T (registers)
//   O^T (D x 8 rows)       += V^T (16 d x 16 keys per m-tile, ldmatrix.trans)
//                             . P^T (the S^T accumulators, bf16, moved into
//                               operand layout with four shuffles)
// A thread of the S^T accumulators holds keys g, g+8 of rows 2c, 2c+1 (g =
// lane/4, c = lane%4): the running max and sum of a row live in the 8 lanes
// that share c.  K and V rows of a step are gathered by slot with 16-byte
// cp.async into a ring of PipeCfg<D>::STAGES stages (one fewer steps in
// flight) whose rows are padded by 16 B, so ldmatrix reads all 32 banks.
// The max is rescaled lazily: O and the sum are rescaled only when a row's
// max grows by more than 2^8.
constexpr int kPipeWarps = 6;                    // warps of a CTA in the warp role
constexpr int kSlotBuf = 128;                    // key slots per slot block (x 16 B aligned)
constexpr int kSlotRegs = kSlotBuf / 32;         // slots of a block per lane
template <int D>
struct PipeCfg {
  static constexpr int STAGES = D == 128 ? 4 : 2;     // ring stages per warp
  static constexpr int PITCH = 2 * D + 16;            // shared bytes per K/V row
  static constexpr int STAGE_BYTES = 32 * PITCH;      // 16 K rows, then 16 V rows
  // the ring, then two slot blocks (the one in use and the next)
  static constexpr int WARP_BYTES = STAGES * STAGE_BYTES + 2 * kSlotBuf * 4;
};

// A warp's next warp-role unit, fetched in stages while the current one
// streams, so that the counter, work-item and slot-table round trips are off
// the path: stage 1 takes an index from the counter (lane 0), stage 2 loads
// the item's work words (lane k < 8 holds word k), stage 3 its first block
// of key slots (lane l holds keys l + 32 i).  idx >= n_small_units: none left.
struct NextUnit {
  int idx;  // lane 0 only until stage 2
  int32_t wk;
  int32_t s[kSlotRegs];
  int stage;
  __device__ __forceinline__ int32_t word(int k) const { return __shfl_sync(0xffffffffu, wk, k); }
};

__device__ __forceinline__ void next_unit_step(const TcArgs& a, NextUnit& n) {
  const int lane = threadIdx.x & 31;
  if (n.stage == 0) {
    n.idx = lane == 0 ? atomicAdd(a.unit_counter, 1) : 0;
  } else if (n.stage == 1) {
    n.idx = __shfl_sync(0xffffffffu, n.idx, 0);
    n.wk = 0;
    if (n.idx < a.n_small_units && lane < RX_WORK_WORDS)
      n.wk = __ldg(a.work_small + int64_t(n.idx / (a.hq / a.group)) * RX_WORK_WORDS + lane);
  } else if (n.stage == 2) {
    const int32_t row = n.word(0), kb = n.word(1), kend = n.word(2), grow = n.word(7);
    if (n.idx < a.n_small_units) {
      const int32_t* trow = a.table + int64_t(row) * a.row_stride;
      const int ke = grow > 0 ? min(kend, grow + a.step) : kend;
#pragma unroll
      for (int i = 0; i < kSlotRegs; ++i) {
        const int key = kb + lane + 32 * i;
        n.s[i] = key < ke ? __ldg(trow + key) : -1;
      }
    }
  }
  if (n.stage < 3) ++n.stage;
}

template <int NR, int D>
__device__ __forceinline__ void pipe_unit(const TcArgs& a, uint32_t ring, int32_t* slot_buf,
                                          uint32_t& gstep, const NextUnit& cur, NextUnit& nxt) {
  using Cfg = PipeCfg<D>;
  constexpr int S = Cfg::STAGES;
  constexpr int kRowPitch = Cfg::PITCH;
  constexpr int kStageBytes = Cfg::STAGE_BYTES;
  constexpr int NK = D / 16;  // k-steps of S^T, m-tiles of O^T
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int n_heads_kv = a.hq / a.group;
  const int unit = cur.idx;
  const int kvh = unit - (unit / n_heads_kv) * n_heads_kv;
  const int G = a.group;
  const int32_t w_row = cur.word(0), w_kend = cur.word(2), w_grow = cur.word(7);
  const int32_t* trow = a.table + int64_t(w_row) * a.row_stride;
  const int kb = cur.word(1), member_off = cur.word(3), part_base = cur.word(5),
            n_rows = cur.word(6);
  // a private tail of a multi-step plan ends at its step-0 end + step
  const int ke = w_grow > 0 ? min(w_kend, w_grow + a.step) : w_kend;
  const bf16* kbase = a.kpool + int64_t(kvh) * a.head_stride;
  const bf16* vbase = a.vpool + int64_t(kvh) * a.head_stride;

  // The unit whose chunk holds this step's newest token (the end of a growing
  // private tail) stores that token's K/V row for its KV head first, so no
  // separate store launch is needed; the bulk copies below then see the row.
  if (a.k_new && w_grow > 0 && ke == w_grow + a.step && kb < ke) {
    const int64_t b = a.members[member_off];
    const int64_t sl = a.slots_new[b];
    if (sl >= 1 && sl < a.num_slots) {
      const int half = lane >> 4, ch = lane & 15;  // lanes 0-15: K, 16-31: V
      const bf16* src = (half ? a.v_new : a.k_new) + (b * n_heads_kv + kvh) * D;
      bf16* dst = const_cast<bf16*>(half ? vbase : kbase) + sl * D;
#pragma unroll
      for (int h = 0; h < D / 128; ++h)
        reinterpret_cast<uint4*>(dst)[ch + 16 * h] =
            __ldg(reinterpret_cast<const uint4*>(src) + ch + 16 * h);
    } else {
      atomicOr(&g_tc_error, 1);
    }
    // only this warp reads the row back (cp.async below): order the lanes'
    // stores before those reads within the CTA
    __threadfence_block();
    __syncwarp();
  }

  const int n_steps = ke > kb ? (ke - kb + 15) >> 4 : 0;
  // Key slots go through two shared blocks of kSlotBuf: block b (keys
  // [kb + 128 b, ..)) sits in half b % 2.  Block 0 comes prefetched with the
  // unit; block b + 1 is loaded into registers when block b is stored, and
  // stored when the first step of block b + 1 is issued, so no table read
  // waits.  -1 past the key range; a slot outside the pool is flagged and
  // read as slot 0.
  int32_t blk[kSlotRegs];
  auto store_block = [&](const int32_t (&r)[kSlotRegs], int half) {
#pragma unroll
    for (int i = 0; i < kSlotRegs; ++i) {
      int32_t sl = r[i];
      if (sl < -1 || sl >= a.num_slots) {
        atomicOr(&g_tc_error, 1);
        sl = 0;
      }
      slot_buf[half * kSlotBuf + lane + 32 * i] = sl;
    }
    __syncwarp();
  };
  auto load_block = [&](int base) {
#pragma unroll
    for (int i = 0; i < kSlotRegs; ++i) {
      const int key = kb + base + lane + 32 * i;
      blk[i] = key < ke ? __ldg(trow + key) : -1;
    }
  };
  if (n_steps > 0) {
    store_block(cur.s, 0);
    load_block(kSlotBuf);
  }
  // step st of this unit: 16 K rows and 16 V rows of 2D bytes, gathered by
  // slot with 16-byte cp.async (lane: chunks lane % 16 (+ 16 h) of rows
  // 8 (lane / 16) + i); rows past the key range are zero-filled (P is 0
  // there, and 0 * V must be 0)
  const int r0 = (lane >> 4) * 8;
  const char* ksrc = reinterpret_cast<const char*>(kbase) + (lane & 15) * 16;
  const int64_t v_minus_k = reinterpret_cast<const char*>(vbase) - reinterpret_cast<const char*>(kbase);
  auto issue = [&](int st) {
    const int block = (st * 16) / kSlotBuf;
    if (block > 0 && st * 16 == block * kSlotBuf) {
      store_block(blk, block & 1);
      load_block((block + 1) * kSlotBuf);
    }
    const uint32_t dst = ring + ((gstep + uint32_t(st)) % S) * kStageBytes +
                         uint32_t(r0 * kRowPitch + (lane & 15) * 16);
    const int4* sp = reinterpret_cast<const int4*>(
        slot_buf + ((block & 1) * kSlotBuf + st * 16 - block * kSlotBuf + r0));
    const int4 s0 = sp[0], s1 = sp[1];
    const int32_t sl[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool ok = sl[i] >= 0;
      const char* src = ksrc + int64_t(ok ? sl[i] : 0) * (D * 2);
#pragma unroll
      for (int h = 0; h < D / 128; ++h) {
        rxk::cp_async_16(dst + uint32_t(i * kRowPitch + 256 * h), src + 256 * h, ok);
        rxk::cp_async_16(dst + uint32_t((16 + i) * kRowPitch + 256 * h), src + 256 * h + v_minus_k,
                         ok);
      }
    }
  };

  float o[NR][NK][4];
#pragma unroll
  for (int nt = 0; nt < NR; ++nt)
#pragma unroll
    for (int mt = 0; mt < NK; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
  float m_ref[NR][2], l_run[NR][2];
#pragma unroll
  for (int nt = 0; nt < NR; ++nt) {
    m_ref[nt][0] = m_ref[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }

#pragma unroll 1
  for (int p = 0; p < S - 1; ++p) {
    if (p < n_steps) issue(p);
    rxk::cp_async_commit();
  }

  // Q^T operand, loaded while the first steps' keys are in flight: n-tile nt,
  // k-step kk: (d 16kk + 2c, +1 | 16kk + 2c + 8, +9) of row nt*8 + g
  uint32_t qb[NR][NK][2];
#pragma unroll
  for (int nt = 0; nt < NR; ++nt) {
    const int r = nt * 8 + g;
    const bool ok = r < n_rows;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q);
    if (ok) {
      const int u = r / G;
      const int64_t b = a.members[member_off + u];
      qrow = reinterpret_cast<const uint32_t*>(a.q + (b * a.hq + kvh * G + (r - u * G)) * D);
    }
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      qb[nt][kk][0] = ok ? __ldg(qrow + 8 * kk + c) : 0u;
      qb[nt][kk][1] = ok ? __ldg(qrow + 8 * kk + c + 4) : 0u;
    }
  }

  // ldmatrix lane addresses: K (A of S^T, keys x d) and V^T (A of O^T, d x keys)
  const uint32_t k_lane = uint32_t(((lane & 7) + ((lane >> 3) & 1) * 8) * kRowPitch + (lane >> 4) * 16);
  const uint32_t v_lane =
      uint32_t((16 + (lane & 7) + (lane >> 4) * 8) * kRowPitch + ((lane >> 3) & 1) * 16);

#pragma unroll 1
  for (int st = 0; st < n_steps; ++st) {
    // the next unit: index at step 0, work words at step 2, slots at step 4
    if (st == 0 || st == 2 || st == 4) next_unit_step(a, nxt);
    rxk::cp_async_wait<S - 2>();
    __syncwarp();
    const uint32_t stage = ring + ((gstep + uint32_t(st)) % S) * kStageBytes;
    // S^T = K . Q^T, even and odd k-steps in two accumulator chains
    float sacc[NR][4], sodd[NR][4];
#pragma unroll
    for (int nt = 0; nt < NR; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = sodd[nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      uint32_t a0, a1, a2, a3;
      rxk::ldsm_x4(stage + k_lane + uint32_t(kk * 32), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NR; ++nt)
        rxk::mma_bf16((kk & 1) ? sodd[nt] : sacc[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NR; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
    // online softmax over the keys of this step (rows 2c, 2c+1 of each n-tile).
    // The row reference m_ref changes only when some key of the row exceeds it
    // by more than 2^8: each lane tests its own keys, one vote per step, and
    // only then are the row maxima reduced over the 8 lanes of a row and O and
    // the sums rescaled (rare after the first step of a unit).
    const int key0 = kb + st * 16 + g;
    const bool in0 = key0 < ke, in1 = key0 + 8 < ke;
    float x[NR][4];
    bool grow = false;
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) {
      x[nt][0] = in0 ? sacc[nt][0] * a.scale_log2 : -INFINITY;
      x[nt][1] = in0 ? sacc[nt][1] * a.scale_log2 : -INFINITY;
      x[nt][2] = in1 ? sacc[nt][2] * a.scale_log2 : -INFINITY;
      x[nt][3] = in1 ? sacc[nt][3] * a.scale_log2 : -INFINITY;
#pragma unroll
      for (int e = 0; e < 2; ++e)
        grow |= fmaxf(x[nt][e], x[nt][2 + e]) > m_ref[nt][e] + kRescaleThreshold;
    }
    if (__any_sync(0xffffffffu, grow)) {
      float mx[NR][2];
#pragma unroll
      for (int nt = 0; nt < NR; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) mx[nt][e] = fmaxf(x[nt][e], x[nt][2 + e]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int nt = 0; nt < NR; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            mx[nt][e] = fmaxf(mx[nt][e], __shfl_xor_sync(0xffffffffu, mx[nt][e], off));
#pragma unroll
      for (int nt = 0; nt < NR; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (mx[nt][e] > m_ref[nt][e]) {
            const float alpha = rxk::fast_exp2(m_ref[nt][e] - mx[nt][e]);  // 0 from -inf
            m_ref[nt][e] = mx[nt][e];
            l_run[nt][e] *= alpha;
#pragma unroll
            for (int mt = 0; mt < NK; ++mt) {
              o[nt][mt][e] *= alpha;
              o[nt][mt][2 + e] *= alpha;
            }
          }
        }
    }
    uint32_t pk[NR][2];  // (key g | key g+8) of rows 2c, 2c+1 as bf16x2
#pragma unroll
    for (int nt = 0; nt < NR; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float m_use = m_ref[nt][e] == -INFINITY ? 0.f : m_ref[nt][e];
        uint32_t h;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n"
            : "=r"(h)
            : "f"(rxk::fast_exp2(x[nt][2 + e] - m_use)), "f"(rxk::fast_exp2(x[nt][e] - m_use)));
        pk[nt][e] = h;  // low half: key g, high half: key g+8
        l_run[nt][e] += __uint_as_float(h << 16) + __uint_as_float(h & 0xffff0000u);
      }
    // P^T operand for n-tile nt: b0 = (P[key 2c][row g], P[key 2c+1][row g]),
    // b1 = keys 2c+8, 2c+9; key k of row r sits in lane 4k + r/2, half r%2
    uint32_t pb[NR][2];
    const int src1 = 8 * c + (g >> 1), src2 = src1 + 4;
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) {
      const uint32_t v0 = __shfl_sync(0xffffffffu, pk[nt][0], src1);
      const uint32_t v1 = __shfl_sync(0xffffffffu, pk[nt][1], src1);
      const uint32_t w0 = __shfl_sync(0xffffffffu, pk[nt][0], src2);
      const uint32_t w1 = __shfl_sync(0xffffffffu, pk[nt][1], src2);
      const uint32_t s1 = (g & 1) ? v1 : v0;
      const uint32_t s2 = (g & 1) ? w1 : w0;
      pb[nt][0] = __byte_perm(s1, s2, 0x5410);
      pb[nt][1] = __byte_perm(s1, s2, 0x7632);
    }
    // O^T += V^T . P^T
#pragma unroll
    for (int mt = 0; mt < NK; ++mt) {
      uint32_t a0, a1, a2, a3;
      rxk::ldsm_x4_t(stage + v_lane + uint32_t(mt * 32), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) rxk::mma_bf16(o[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
    if (st + S - 1 < n_steps) issue(st + S - 1);
    rxk::cp_async_commit();
  }
  rxk::cp_async_wait<0>();
  __syncwarp();
  gstep += uint32_t(n_steps);

  // write the partial (o, lse) of rows nt*8 + 2c + e
#pragma unroll
  for (int nt = 0; nt < NR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[nt][e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int r = nt * 8 + 2 * c + e;
      if (r >= n_rows) continue;
      const int uu = r / G;
      const int head = kvh * G + (r - uu * G);
      const int64_t part = int64_t(part_base) + uu;
      float* dst = a.ws_o + (part * a.hq + head) * D;
      const float inv = l > 0.f ? 1.f / l : 0.f;  // an empty chunk: zero partial, lse -inf
#pragma unroll
      for (int mt = 0; mt < NK; ++mt) {
        dst[16 * mt + g] = o[nt][mt][e] * inv;
        dst[16 * mt + g + 8] = o[nt][mt][2 + e] * inv;
      }
      if (g == 0) a.ws_lse[part * a.hq + head] = l > 0.f ? m_ref[nt][e] * kLn2 + logf(l) : -INFINITY;
    }
}

// One launch per decode step, at most one CTA per SM.  CTAs [w, w + n_tc_ctas)
// (w = n_warp_first) first run the tensor-core tile of one segment chunk with
// more than 16 query rows (CTA w + c: item c / Hkv, KV head c % Hkv).  Then
// the first six warps of every CTA take warp-role units (an item of <= 16
// rows and one KV head) from a shared counter, heaviest first, until none is
// left; so the SMs of finished tiles join the warp-role work.  When the tiles
// alone fill more than one wave, the w CTAs before them take warp-role units
// from the start, so the streaming of private tails (bound by HBM) runs
// beside the first wave of tiles (bound by the tensor core and the
// exponentials) instead of after it.  The counter starts at 0 and the merge
// after this kernel resets it.  Launched with programmatic stream
// serialization: the merge that follows may launch early, and this kernel waits
// (griddepcontrol.wait) for the previous kernels on the stream before it
// touches what they wrote or read.
template <int D>
struct Fused {
  static constexpr int THREADS = kThreads3;
  static constexpr int TILE_BYTES = Layout3<D>::BYTES;
  static constexpr int PIPE_BYTES = kPipeWarps * PipeCfg<D>::WARP_BYTES + 1024;
  static constexpr int SMEM = TILE_BYTES > PIPE_BYTES ? TILE_BYTES : PIPE_BYTES;
  static_assert(SMEM <= 227 * 1024, "fused decode CTA fits in shared memory");
};

template <int D>
__global__ void __launch_bounds__(Fused<D>::THREADS, 1)
    decode_fused_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
  using Cfg = PipeCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  rxk::griddep_launch_dependents();
  const int cta = int(blockIdx.x) - a.n_warp_first;
  if (cta >= 0 && cta < a.n_tc_ctas) {
    const int hkv = a.hq / a.group;
    tc_tile3<D, true>(a, &tmk, &tmv, smem_raw, cta / hkv, cta - (cta / hkv) * hkv);
  }
  if (threadIdx.x >= kPipeWarps * 32) return;  // the warp role uses the first six warps
  // tiles_leave: in a run of steps a tile CTA leaves its SM to the next
  // step's tiles, which start there at once (early inputs) while this step's
  // warp-role units still stream on the other SMs
  if (a.tiles_leave && cta >= 0 && cta < a.n_tc_ctas) return;
  rxk::griddep_wait();
  // warp role: this warp's ring and slot buffer
  const uint32_t raw = rxk::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int warp = int(threadIdx.x >> 5);
  const int lane = int(threadIdx.x & 31);
  const uint32_t ring = base + uint32_t(warp * Cfg::WARP_BYTES);
  int32_t* slot_buf = reinterpret_cast<int32_t*>(smem_raw + (base - raw) + warp * Cfg::WARP_BYTES +
                                                 Cfg::STAGES * Cfg::STAGE_BYTES);  // [2][kSlotBuf]
  uint32_t gstep = 0;
  NextUnit cur, nxt;
  cur.stage = 0;
  while (cur.stage < 3) next_unit_step(a, cur);
  while (cur.idx < a.n_small_units) {
    nxt.stage = 0;
    const int rows = cur.word(6);
    if (rows <= 8) {
      pipe_unit<1, D>(a, ring, slot_buf, gstep, cur, nxt);
    } else if constexpr (D == 128) {
      pipe_unit<2, D>(a, ring, slot_buf, gstep, cur, nxt);
    } else if (lane == 0) {
      atomicOr(&g_tc_error, 1);  // the plan gives head_dim 256 no such item
    }
    while (nxt.stage < 3) next_unit_step(a, nxt);  // short units: the rest now
    cur = nxt;
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once per process (a function-
// local static is initialised exactly once, whichever thread gets there).
EncodeTiled encode_fn() {
  static const EncodeTiled fn = []() -> EncodeTiled {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiled>(p);
    return nullptr;
  }();
  return fn;
}

// Tensor map over a whole pool [L * Hkv * num_slots rows][D] of bf16, box of
// 64 columns x BN rows, 128-byte swizzle (the shared-memory tile layout);
// false if it cannot be encoded or the pool has 2^31 rows or more.
bool make_pool_map(CUtensorMap* m, const void* pool, const rx_pool_desc* d, int BN) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  // TMA row coordinates are 32-bit signed
  if (int64_t(d->num_layers) * d->num_kv_heads * d->num_slots > INT32_MAX) return false;
  const cuuint64_t dims[2] = {cuuint64_t(d->head_dim),
                              cuuint64_t(d->num_layers) * d->num_kv_heads * d->num_slots};
  const cuuint64_t strides[1] = {cuuint64_t(d->head_dim) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(BN)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the pools last used on this thread (K and V of one pool
// descriptor): encoding them is host work repeated on every launch otherwise.
struct PoolMaps {
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t num_slots = 0;
  int32_t layers = 0, heads = 0, dim = 0, box_rows = 0;
  CUtensorMap mk, mv;
};

bool pool_maps(const rx_pool_desc* d, int BN, const CUtensorMap** mk, const CUtensorMap** mv) {
  thread_local PoolMaps cache[4];
  thread_local int next = 0;
  for (PoolMaps& c : cache) {
    if (c.k == d->k_pool && c.v == d->v_pool && c.num_slots == d->num_slots &&
        c.layers == d->num_layers && c.heads == d->num_kv_heads && c.dim == d->head_dim &&
        c.box_rows == BN) {
      *mk = &c.mk;
      *mv = &c.mv;
      return true;
    }
  }
  PoolMaps& c = cache[next];
  next = (next + 1) & 3;
  c.k = nullptr;
  if (!make_pool_map(&c.mk, d->k_pool, d, BN) || !make_pool_map(&c.mv, d->v_pool, d, BN))
    return false;
  c.k = d->k_pool;
  c.v = d->v_pool;
  c.num_slots = d->num_slots;
  c.layers = d->num_layers;
  c.heads = d->num_kv_heads;
  c.dim = d->head_dim;
  c.box_rows = BN;
  *mk = &c.mk;
  *mv = &c.mv;
  return true;
}

// A kernel's dynamic shared-memory limit is an attribute of the kernel in
// the current device's context: it is raised once per device (any thread
// may do it first; setting it twice is harmless).
constexpr int kMaxDevices = 64;

template <typename K>
rx_status ensure_smem(std::atomic<bool> (&done)[kMaxDevices], K* kernel, int bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return rx_internal::set_error(RX_ERR_CUDA, "no usable current device");
  if (done[dev].load(std::memory_order_acquire)) return RX_OK;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();  // not left for a later launch check to report
    static thread_local char buf[160];
    snprintf(buf, sizeof(buf), "raising a kernel's shared-memory limit: %s",
             cudaGetErrorString(e));
    return rx_internal::set_error(RX_ERR_CUDA, buf);
  }
  done[dev].store(true, std::memory_order_release);
  return RX_OK;
}

template <int D>
rx_status launch_extend(TcArgs a, const rx_pool_desc* pool, int32_t layer, unsigned gx,
                        unsigned gy, cudaStream_t s) {
  using Lo = Layout3<D>;
  static std::atomic<bool> configured[kMaxDevices];
  const rx_status cs = ensure_smem(configured, attn_tc3_kernel<D>, Lo::BYTES);
  if (cs != RX_OK) return cs;
  const CUtensorMap *tmk, *tmv;
  if (!pool_maps(pool, Lo::BN, &tmk, &tmv))
    return rx_internal::set_error(RX_ERR_CUDA, "could not encode the pool's TMA tensor maps");
  a.tma_row_base = int64_t(layer) * pool->num_kv_heads * pool->num_slots;
  a.tma_head_rows = pool->num_slots;
  attn_tc3_kernel<D><<<dim3(gx * gy), kThreads3, Lo::BYTES, s>>>(a, *tmk, *tmv);
  return rx_internal::launch_status("extend attention (tcgen05)");
}

}  // namespace

namespace rx_internal {

int32_t tc_error_flags(bool clear) {
  int32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v));
  if (clear && v) {
    int32_t z = 0;
    cudaMemcpyToSymbol(g_tc_error, &z, sizeof(z));
  }
  return v;
}

rx_status decode_fused(const rx_pool_desc* pool, int32_t layer, const void* d_q,
                       int32_t num_q_heads, const int32_t* d_req_to_token, int64_t row_stride,
                       const int32_t* d_work_small, int64_t n_small, const int32_t* d_work_tc,
                       int64_t n_tc, const int32_t* d_members, float scale, float* ws_o,
                       float* ws_lse, int32_t* unit_counter, int step, const void* k_new,
                       const void* v_new, const int32_t* slots_new, cudaStream_t stream,
                       bool early_inputs) {
  const int D = pool->head_dim;
  if (D != 128 && D != 256) return set_error(RX_ERR_INVALID, "decode needs head_dim 128 or 256");
  const int64_t hkv = pool->num_kv_heads;
  const int64_t small_units = n_small * hkv;
  const int64_t tc_ctas = n_tc * hkv;
  // the tiles plus CTAs for the warp-role units: when everything fits in one
  // wave, enough of them for every unit (after the tiles); otherwise up to a
  // quarter of the SMs, placed before the tiles so that they start at once
  const int64_t sms = rx_internal::sm_count();
  const int64_t unit_ctas = (small_units + kPipeWarps - 1) / kPipeWarps;
  int64_t warp_first = 0, ctas = tc_ctas;
  if (tc_ctas + unit_ctas <= sms)
    ctas = tc_ctas + unit_ctas;
  else if (tc_ctas >= sms)
    warp_first = std::min<int64_t>(unit_ctas, (sms + 3) / 4);
  else
    ctas = sms;
  ctas += warp_first;
  if (ctas == 0) return RX_OK;
  if (ctas > INT32_MAX) return set_error(RX_ERR_INVALID, "decode plan too large for one launch");
  TcArgs a{};
  a.q = static_cast<const bf16*>(d_q);
  const int64_t layer_off = int64_t(layer) * hkv * pool->num_slots * D;
  a.kpool = static_cast<const bf16*>(pool->k_pool) + layer_off;
  a.vpool = static_cast<const bf16*>(pool->v_pool) + layer_off;
  a.head_stride = pool->num_slots * D;
  a.num_slots = pool->num_slots;
  a.table = d_req_to_token;
  a.row_stride = row_stride;
  a.hq = num_q_heads;
  a.group = num_q_heads / int(hkv);
  a.scale_log2 = scale * kLog2e;
  a.work = d_work_tc;
  a.members = d_members;
  a.ws_o = ws_o;
  a.ws_lse = ws_lse;
  a.work_small = d_work_small;
  a.n_small_units = int(small_units);
  a.n_tc_ctas = int(tc_ctas);
  a.n_warp_first = int(warp_first);
  a.unit_counter = unit_counter;
  a.early_inputs = early_inputs ? 1 : 0;
  // with three times as many warp-role CTAs as tile CTAs (few, long tiles
  // beside many units), the tiles need not help with the units
  a.tiles_leave = early_inputs && ctas - tc_ctas >= 3 * tc_ctas ? 1 : 0;
  a.step = step;
  a.k_new = static_cast<const bf16*>(k_new);
  a.v_new = static_cast<const bf16*>(v_new);
  a.slots_new = slots_new;
  a.tma_row_base = int64_t(layer) * hkv * pool->num_slots;
  a.tma_head_rows = pool->num_slots;
  static std::atomic<bool> configured128[kMaxDevices], configured256[kMaxDevices];
  const rx_status cs =
      D == 128 ? ensure_smem(configured128, decode_fused_kernel<128>, Fused<128>::SMEM)
               : ensure_smem(configured256, decode_fused_kernel<256>, Fused<256>::SMEM);
  if (cs != RX_OK) return cs;
  const CUtensorMap *tmk, *tmv;
  if (!pool_maps(pool, D == 128 ? 128 : 64, &tmk, &tmv))
    return set_error(RX_ERR_CUDA, "could not encode the pool's TMA tensor maps");
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(ctas));
  cfg.blockDim = dim3(unsigned(D == 128 ? Fused<128>::THREADS : Fused<256>::THREADS));
  cfg.dynamicSmemBytes = D == 128 ? Fused<128>::SMEM : Fused<256>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128)
    cudaLaunchKernelEx(&cfg, decode_fused_kernel<128>, a, *tmk, *tmv);
  else
    cudaLaunchKernelEx(&cfg, decode_fused_kernel<256>, a, *tmk, *tmv);
  return launch_status("decode attention (fused)");
}

rx_status extend_attention_tc(const rx_pool_desc* pool, int32_t layer, const void* d_q,
                              int32_t num_q_heads, const int32_t* d_req_to_token,
                              int64_t row_stride, const int32_t* d_req_rows,
                              const int32_t* d_prefix_len, const int32_t* d_qo_indptr,
                              const int32_t* d_tile_indptr, int32_t R, int64_t num_tiles,
                              float scale, float* d_out, float* d_lse, cudaStream_t stream) {
  const int D = pool->head_dim;
  TcArgs a{};
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
  a.req_rows = d_req_rows;
  a.prefix_len = d_prefix_len;
  a.qo_indptr = d_qo_indptr;
  a.tile_indptr = d_tile_indptr;
  a.num_req = R;
  a.num_tiles = int(num_tiles);
  // heads interleaved (the heavy row tiles of every head first, a short
  // tail) for up to kExtendInterleaveWaves waves of CTAs, or when a
  // request's keys over all heads are small enough to stay in L2 while its
  // row tiles run (row_stride bounds a request's keys); otherwise
  // head-major, so the CTAs in flight read one head's long key ranges
  const int64_t kv_row_bytes = row_stride * pool->num_kv_heads * int64_t(D) * 4;
  a.heads_interleaved =
      num_tiles * pool->num_kv_heads <= int64_t(kExtendInterleaveWaves) * rx_internal::sm_count() ||
      kv_row_bytes <= kExtendInterleaveKvBytes;
  a.out = d_out;
  a.lse = d_lse;
  if (D == 128)
    return launch_extend<128>(a, pool, layer, unsigned(num_tiles), pool->num_kv_heads, stream);
  return launch_extend<256>(a, pool, layer, unsigned(num_tiles), pool->num_kv_heads, stream);
}

}  // namespace rx_internal
