// Forward pass of blocked GQA flash attention on sm_103a.
//
// One CTA owns one Q tile: the G query heads of one kv head packed into 128
// rows (row r = g * (128/G) + i, position t = t0 + i), loaded once by TMA.  It
// sweeps the non-empty KV tiles of 128 keys with the online softmax of
// "Chunked attention" (danielwatson6.github.io/fa/fa.html): running max m,
// denominator l, accumulator O rescaled when m moves, O / l at the end; the
// accumulator never leaves the chip and the T x S weights never reach memory
// ("Optimizing the kernel": carries kept on chip, bf16 output).
//
// Roles (warp specialisation, 192 threads):
//   warps 0-3  softmax: thread r owns TMEM lane r = packed row r
//   warp  4    TMA producer (lane 0): Q once, then K/V in 16 KB chunks
//   warp  5    MMA issuer (lane 0) and TMEM owner
//
// Tensor memory (512 columns): O accumulator in columns [0, H); two S buffers
// of 128 fp32 columns at 256 and 384.  P (bf16, 2 per column) overwrites the
// first 64 columns of its S buffer and is the A operand of O += P V.
//
// Shared memory: Q tile (H/64 chunks of [128 rows x 128 B]), a ring of
// kSlots chunks of [128 keys x 64 dims] bf16 fed by TMA with 128-byte swizzle
// (one copy per fwd_copy_chunks(H) consecutive chunks of a K or V tile),
// the per-tile schedule and the mbarriers.
#include <cuda_bf16.h>
#include "block_mask.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 192;
constexpr int kSlots = 8;
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

template <int H>
struct FwdSmem {
  static constexpr int HC = H / 64;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t ring_off = HC * kChunkBytes;
  static constexpr uint32_t tiles_off = ring_off + kSlots * kChunkBytes;   // uint16 schedule
  static constexpr uint32_t cls_off = tiles_off + kMaxKvTiles * 2;         // uint8 classes
  static constexpr uint32_t runs_off = cls_off + kMaxKvTiles;               // uint8 segment runs
  static constexpr uint32_t bar_off = runs_off + kMaxKvTiles;
  // barriers: q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2], pv_done[2], teardown
  static constexpr int n_bars = 1 + 2 * kSlots + 7;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;  // tmem slot, abort, count, qrange
  static constexpr uint32_t bytes = misc_off + 64;
  static constexpr uint32_t alloc = bytes + 1024;  // room to align the base to 1024
};

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t empty(int s) const { return base + 8 * (1 + kSlots + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 2 * kSlots + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (3 + 2 * kSlots + b); }
  __device__ uint32_t pv_done(int b) const { return base + 8 * (5 + 2 * kSlots + b); }
  __device__ uint32_t teardown() const { return base + 8 * (7 + 2 * kSlots); }
};

// All lanes of a warp agree on the outcome of a bounded wait, so the
// warp-collective TMEM accesses that follow are executed by all or none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  const bool ok = mbar_wait(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// K/V chunks travel through the ring in the order the MMA warp consumes them:
// K(0), K(1), V(0), K(2), V(1), ..., K(N-1), V(N-2), V(N-1).  Unit u holds the
// H/64 chunks of one K or V tile; chunk c of unit u has sequence number u*HC+c.
__device__ __forceinline__ uint32_t unit_k(int n) { return n == 0 ? 0u : (uint32_t)(2 * n - 1); }
__device__ __forceinline__ uint32_t unit_v(int n, int n_tiles) {
  return (uint32_t)min(2 * n + 2, 2 * n_tiles - 1);
}

// Tile classes of the lazy mask.
enum : uint8_t { TILE_EMPTY = 0, TILE_FULL = 1, TILE_PARTIAL = 2 };

// One KV tile of the online softmax for packed row r (TMEM lane r): wait for
// S(N) (global tile counter N: buffer N & 1), apply the lazy mask on PARTIAL
// tiles, update the running max m_ref / denominator l (rescaling O, after
// O += P V of tile N - 1, only when m moved by more than 2^8), write P (bf16)
// over the first 64 columns of the S buffer and signal p_full.  n is the tile's
// index within its Q tile (n == 0 starts the row).  O lives in TMEM columns
// [o_col, o_col + H).  Returns false when a bounded wait gave up.
template <int H>
__device__ __forceinline__ bool softmax_tile(const FwdArgs& a, uint32_t tmem, uint32_t lane_base,
                                             uint16_t entry, uint8_t runs, int n, int N, int t, int g,
                                             bool valid, int my_seg, int b, int kh, const Bars& bars,
                                             const Abort& ab, float& m_ref, float& l,
                                             uint32_t o_col = 0) {
  const int j = entry & 0x7fff;
  const bool partial = (entry & 0x8000) != 0;
  const int off = a.S - a.T;
  const bool segs = a.seg_q != nullptr;
  if (!warp_wait(bars.s_full(N & 1), (N >> 1) & 1, ab)) return false;
  tc_fence_after();
  const uint32_t s_col = 256 + 128 * (N & 1);
  uint32_t sv[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + s_col + c * 32, sv[c]);
  tmem_wait_ld();
  float* s = reinterpret_cast<float*>(&sv[0][0]);
  if (partial) {
    // Keys kept by the causal and range limits form [klo, khi); with segment
    // ids in at most two runs (`runs` < kRunsGeneral) the row's id selects one
    // run, which narrows the same range.  The range becomes four 32-bit keep
    // words, one select per score.  Other segment layouts compare ids one by one.
    const int s0 = j * kKvRows;
    const int n_keys = min(kKvRows, a.S - s0);
    int klo = 0, khi = n_keys;
    if (a.causal) khi = min(khi, t + off - s0 + 1);
    bool per_key = false;
    if (segs) {
      if (runs != kRunsGeneral) {
        const int32_t* ids = a.seg_kv + (long)b * a.S + s0;
        if (my_seg == __ldg(ids)) khi = min(khi, (int)runs);
        else if (runs < n_keys && my_seg == __ldg(ids + n_keys - 1)) klo = runs;
        else khi = 0;
      } else {
        per_key = true;
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t keep = range_bits(klo - 32 * w, khi - 32 * w);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!((keep >> i) & 1u)) s[32 * w + i] = -INFINITY;
    }
    if (per_key) {
      // every thread reads the same 512 B of key ids: served by L1 broadcast
      const int32_t* ids = a.seg_kv + (long)b * a.S + s0;
      if ((a.S & 3) == 0 && s0 + 128 <= a.S) {  // aligned and in range
        const int4* kid = reinterpret_cast<const int4*>(ids);
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) {
          const int4 v = __ldg(kid + c4);
          if (v.x != my_seg) s[4 * c4 + 0] = -INFINITY;
          if (v.y != my_seg) s[4 * c4 + 1] = -INFINITY;
          if (v.z != my_seg) s[4 * c4 + 2] = -INFINITY;
          if (v.w != my_seg) s[4 * c4 + 3] = -INFINITY;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (s0 + c < a.S && __ldg(ids + c) != my_seg) s[c] = -INFINITY;
      }
    }
    if (a.bm.cls != nullptr && valid) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t bits = bm_row_word(a.bm, kh, a.G, g, t, j, w);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (!((bits >> i) & 1u)) s[32 * w + i] = -INFINITY;
      }
    }
  }
  // Row max with 8 independent partial maxima (short dependency chains).
  float pm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pm[i] = s[i];
#pragma unroll
  for (int c = 8; c < 128; c += 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) pm[i] = fmaxf(pm[i], s[c + i]);
  }
  const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                         fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
  const float m_tile = mx * kLog2e;
  float alpha = 1.f;
  bool rescale = false;
  if (n == 0) {
    m_ref = m_tile;
  } else if (m_tile > m_ref + kRescaleThreshold) {
    alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_tile);
    m_ref = m_tile;
    rescale = true;
  }
  const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
  // O must be rescaled before O += P V of this tile; it holds every earlier tile.
  if (__any_sync(0xffffffffu, rescale)) {
    if (!warp_wait(bars.pv_done((N - 1) & 1), ((N - 1) >> 1) & 1, ab)) return false;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < H; c += 32) {
      uint32_t ov[32];
      tmem_ld32(tmem + lane_base + o_col + c, ov);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
      tmem_st32(tmem + lane_base + o_col + c, ov);
    }
  }
  // P = exp2(S log2e - m) in two halves of 64 keys; bf16 pairs overwrite the
  // first 64 columns of this tile's S buffer (already read into registers).
  float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    uint32_t pk[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float p0 = fast_exp2(fmaf(s[64 * hf + 2 * c], kLog2e, -m_use));
      const float p1 = fast_exp2(fmaf(s[64 * hf + 2 * c + 1], kLog2e, -m_use));
      ps[c & 3] += p0 + p1;
      pk[c] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tmem + lane_base + s_col + 32 * hf, pk);
  }
  l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(bars.p_full(N & 1));
  return true;
}

// O / l of packed row r in bf16 into a Q-shaped shared-memory tile (H/64
// chunks of [128 rows x 128 B], 128-byte swizzle), ready for TMA stores.  O is
// read from TMEM columns [o_col, o_col + H) when `have`, else zeros are written.
template <int H>
__device__ __forceinline__ void stage_o_row(uint8_t* q_tile, uint32_t tmem, uint32_t lane_base,
                                            uint32_t o_col, int r, bool have, float inv) {
#pragma unroll 1
  for (int c = 0; c < H; c += 32) {
    uint32_t ov[32];
    if (have) {
      tmem_ld32(tmem + lane_base + o_col + c, ov);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) ov[i] = 0;
    }
    uint4 pkd[4];
    uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pw[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
    uint8_t* chunk = q_tile + (c / 64) * kChunkBytes;
    const uint32_t u0 = (c % 64) / 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(chunk + sw128_offset(r, u0 + i)) = pkd[i];
  }
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdArgs a) {
  using L = FwdSmem<H>;
  constexpr int HC = L::HC;
  constexpr int CC = fwd_copy_chunks(H);  // chunks per K/V copy
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(sm);

  uint16_t* tiles = reinterpret_cast<uint16_t*>(sm + L::tiles_off);
  uint8_t* cls = sm + L::cls_off;
  uint8_t* runs = sm + L::runs_off;  // per KV tile j (segment ids only)
  Bars bars{sbase + L::bar_off};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc_off + 4);
  int* n_tiles_s = reinterpret_cast<int*>(sm + L::misc_off + 8);
  int* qrange = reinterpret_cast<int*>(sm + L::misc_off + 16);
  const Abort ab{abort_flag, a.wait_limit_ns, a.err};

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int Tb = kRows / a.G;                      // positions per Q tile
  // Flat grid, Q-tile major: the latest (causally heaviest) Q tiles of every
  // (batch, kv head) are dispatched first.
  const int BKn = a.B * a.K;
  const int qt = a.n_qtiles - 1 - (int)(blockIdx.x / BKn);
  const int bk = (int)(blockIdx.x % BKn);
  const int b = bk / a.K;
  const int t0 = qt * Tb;
  const int n_valid = min(Tb, a.T - t0);   // positions of this tile below T
  const int off = a.S - a.T;               // causal keeps s <= t + off
  const int n_kv_all = (a.S + kKvRows - 1) / kKvRows;
  const bool segs = a.seg_q != nullptr;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full(i), 1);
      mbar_init(bars.p_full(i), kRows);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.teardown(), 1);
    fence_barrier_init();
    // Every CTA with work needs its Q tile: start the copy before the
    // schedule is built, so its latency overlaps the tile classification.
    mbar_arrive_expect_tx(bars.q_full(), HC * kChunkBytes);
    for (int c = 0; c < HC; ++c)
      tma_load_4d(sbase + L::q_off + c * kChunkBytes, &a.tm_q, bars.q_full(), c * 64, t0, 0, bk);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 4) {
    prefetch_tmap(&a.tm_q);
    prefetch_tmap(&a.tm_k);
    prefetch_tmap(&a.tm_v);
  }

  // KV tiles the causal mask can reach: keys s <= t_last + off.
  int n_kv = n_kv_all;
  if (a.causal) {
    const int lim = t0 + n_valid - 1 + off;
    n_kv = lim < 0 ? 0 : min(n_kv_all, lim / kKvRows + 1);
  }

  // Segment range of this Q tile (ids of its Tb positions).
  if (segs && warp == 0) {
    int mn = INT_MAX, mx = INT_MIN;
    for (int i = lane; i < n_valid; i += 32) {
      int v = a.seg_q[(long)b * a.T + t0 + i];
      mn = min(mn, v);
      mx = max(mx, v);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) { qrange[0] = mn; qrange[1] = mx; }
  }
  __syncthreads();

  // Classify every reachable KV tile (lazy mask: only per-tile id ranges).
  for (int j = warp; j < n_kv; j += kThreads / 32) {
    uint8_t c = TILE_FULL;
    const int s_last = min((j + 1) * kKvRows, a.S) - 1;
    if (a.causal && s_last > t0 + off) c = TILE_PARTIAL;  // crosses the diagonal
    if ((j + 1) * kKvRows > a.S) c = TILE_PARTIAL;         // ragged last tile
    if (segs) {
      // 4 keys per lane; keys past S repeat the last key's id (no effect on the
      // range, no extra run)
      int mn = INT_MAX, mx = INT_MIN, v[4];
      for (int e = 0; e < 4; ++e) {
        v[e] = a.seg_kv[(long)b * a.S + min(j * kKvRows + lane * 4 + e, s_last)];
        mn = min(mn, v[e]);
        mx = max(mx, v[e]);
      }
      mn = __reduce_min_sync(0xffffffffu, mn);
      mx = __reduce_max_sync(0xffffffffu, mx);
      const int qmn = qrange[0], qmx = qrange[1];
      if (mx < qmn || mn > qmx) c = TILE_EMPTY;
      else if (!(mn == mx && qmn == qmx && mn == qmn)) c = TILE_PARTIAL;
      // where the id changes, if it changes at most once
      int changes = (v[1] != v[0]) + (v[2] != v[1]) + (v[3] != v[2]);
      int pos = v[1] != v[0] ? 4 * lane + 1 : v[2] != v[1] ? 4 * lane + 2 : v[3] != v[2] ? 4 * lane + 3 : kKvRows;
      const int prev = __shfl_up_sync(0xffffffffu, v[3], 1);
      if (lane > 0 && v[0] != prev) { ++changes; pos = 4 * lane; }
      changes = __reduce_add_sync(0xffffffffu, changes);
      pos = __reduce_min_sync(0xffffffffu, pos);
      if (lane == 0) runs[j] = changes == 0 ? (uint8_t)kKvRows : changes == 1 ? (uint8_t)pos : kRunsGeneral;
    }
    if (a.bm.cls != nullptr)  // the Q tile lies inside one 128-position mask block
      c = (uint8_t)class_and(c, bm_tile_class(a.bm, bk % a.K, a.G, t0 >> 7, j));
    if (lane == 0) cls[j] = c;
  }
  __syncthreads();
  // Compact the non-empty tiles into the schedule (warp 0, ballot prefix sums).
  if (warp == 0) {
    int count = 0;
    for (int j0 = 0; j0 < n_kv; j0 += 32) {
      const int j = j0 + lane;
      const uint8_t c = j < n_kv ? cls[j] : TILE_EMPTY;
      const uint32_t m = __ballot_sync(0xffffffffu, c != TILE_EMPTY);
      if (c != TILE_EMPTY) {
        const int pos = count + __popc(m & ((1u << lane) - 1));
        tiles[pos] = (uint16_t)(j | (c == TILE_PARTIAL ? 0x8000 : 0));
      }
      count += __popc(m);
    }
    if (lane == 0) *n_tiles_s = count;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Split-KV mode: this CTA takes slice blockIdx.z of the schedule.
  const int n_sched = *n_tiles_s;
  const int per_split = (n_sched + a.n_splits - 1) / a.n_splits;
  const int sched_begin = min(n_sched, (int)blockIdx.z * per_split);
  const int n_tiles = min(n_sched, sched_begin + per_split) - sched_begin;
  const uint16_t* sched = tiles + sched_begin;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      uint32_t seq = 0;
      bool ok = true;
      for (int u = 0; u < 2 * n_tiles && ok; ++u) {
        // unit 0: K(0); last unit: V(N-1); odd u: K((u+1)/2); even u: V(u/2 - 1)
        bool is_k;
        int n;
        if (u == 0) { is_k = true; n = 0; }
        else if (u == 2 * n_tiles - 1) { is_k = false; n = n_tiles - 1; }
        else if (u & 1) { is_k = true; n = (u + 1) / 2; }
        else { is_k = false; n = u / 2 - 1; }
        const int j = sched[n] & 0x7fff;
        const CUtensorMap* m = is_k ? &a.tm_k : &a.tm_v;
        // The unit's HC chunks sit in consecutive slots (kSlots is a multiple
        // of HC).  Each copy fills CC of them and completes on the first one's
        // barrier, once every chunk's previous reader has released its slot.
        for (int cc = 0; cc < HC && ok; cc += CC, seq += CC) {
          for (int c = 0; c < CC && ok; ++c) {
            const uint32_t sq = seq + c;
            if (sq >= kSlots && !mbar_wait(bars.empty(sq % kSlots), ((sq / kSlots) - 1) & 1, ab)) ok = false;
          }
          if (!ok) break;
          const int slot = seq % kSlots;
          mbar_arrive_expect_tx(bars.full(slot), CC * kChunkBytes);
          tma_load_4d(sbase + L::ring_off + slot * kChunkBytes, m, bars.full(slot), 0, j * kKvRows, cc, bk);
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        const uint32_t first = seq > kSlots ? seq - kSlots : 0;
        for (uint32_t s = first; s < seq; s += CC)  // one copy per CC chunks, on its first slot
          mbar_wait_teardown(bars.full(s % kSlots), (s / kSlots) & 1, a.wait_limit_ns);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T
      constexpr uint32_t id_o = idesc_bf16(128, H, false, true);     // O += P V (N = H)
      // Operand descriptors, built once and advanced by byte offsets.
      const uint64_t dq0 = sdesc_sw128(sbase + L::q_off, 16, 1024);        // Q, K-major
      const uint64_t dk0 = sdesc_sw128(sbase + L::ring_off, 16, 1024);     // K chunk, K-major
      const uint64_t dv0 = sdesc_sw128(sbase + L::ring_off, kChunkBytes, 1024);  // V, MN-major
      bool ok = mbar_wait(bars.q_full(), 0, ab);
      auto issue_pv = [&](int n) -> bool {
        if (!mbar_wait(bars.p_full(n & 1), (n >> 1) & 1, ab)) return false;
        const uint32_t seq0 = unit_v(n, n_tiles) * HC;
        const int slot0 = seq0 % kSlots;  // the unit's HC chunks sit in consecutive slots
        for (int c = 0; c < HC; c += CC)  // every copy of the V tile
          if (!mbar_wait(bars.full(slot0 + c), (seq0 / kSlots) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t p_col = 256 + 128 * (n & 1);
        const uint64_t bv = sdesc_add(dv0, slot0 * kChunkBytes);
#pragma unroll
        for (int kk = 0; kk < kKvRows / 16; ++kk)
          mma_ts(tmem, tmem + p_col + kk * 8, sdesc_add(bv, kk * 2048), id_o,
                 (n > 0 || kk > 0) ? 1u : 0u);
        for (int c = 0; c < HC; ++c) mma_commit(bars.empty(slot0 + c));
        mma_commit(bars.pv_done(n & 1));
        return true;
      };
      for (int n = 0; n < n_tiles && ok; ++n) {
        // S buffer n&1 held S(n-2), read by the softmax warps before they signalled
        // P(n-2), and P(n-2), read by O += P V of tile n-2, which this thread issued
        // before S(n): tcgen05.mma ops of one thread execute in issue order.
        const uint32_t s_col = 256 + 128 * (n & 1);
        const uint32_t seq0 = unit_k(n) * HC;
        const int slot0 = seq0 % kSlots;
        for (int c = 0; c < HC && ok; ++c) {
          if (!mbar_wait(bars.full(slot0 + c - c % CC), (seq0 / kSlots) & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a = sdesc_add(dq0, c * kChunkBytes);
          const uint64_t bk_ = sdesc_add(dk0, (slot0 + c) * kChunkBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + s_col, sdesc_add(a, kk * 32), sdesc_add(bk_, kk * 32), id_s,
                   (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bars.empty(slot0 + c));
        }
        if (!ok) break;
        mma_commit(bars.s_full(n & 1));
        if (n >= 1 && !issue_pv(n - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) {
        // Wait (bounded) for every MMA this thread issued before TMEM is freed.
        mma_commit(bars.teardown());
        mbar_wait_teardown(bars.teardown(), 0, a.wait_limit_ns);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int r = tid;  // TMEM lane == packed row
    const int g = r / Tb;
    const int t = t0 + (r - g * Tb);
    const bool valid = t < a.T;  // rows past T (ragged last tile) are computed, not stored
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int my_seg = (segs && valid) ? a.seg_q[(long)b * a.T + t] : 0;
    float m_ref = -INFINITY;  // running max, log2 units
    float l = 0.f;            // running denominator (relative to m_ref)
    bool ok = true;
    for (int n = 0; n < n_tiles; ++n) {
      if (!softmax_tile<H>(a, tmem, lane_base, sched[n], segs ? runs[sched[n] & 0x7fff] : kRunsGeneral,
                           n, n, t, g, valid, my_seg, b, bk % a.K,
                           bars, ab, m_ref, l)) {
        ok = false;
        break;
      }
    }
    // ------------------------------------------------------------ epilogue
    // O / l in bf16 is staged in the Q tile's shared memory (free: every MMA
    // has completed) in the same swizzled layout the Q box arrived in, then
    // written by TMA stores.
    const long row = ((long)bk * a.G + g) * a.T + t;
    const bool have = n_tiles > 0 && ok &&
                      warp_wait(bars.pv_done((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, ab);
    if (have) tc_fence_after();
    const float inv = (have && l > 0.f) ? 1.f / l : 0.f;
    const float lse_row = (have && l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
    if (a.n_splits > 1) {
      // Split-KV: this split's normalised partial output (fp32) and lse; the
      // combine kernel merges the splits with weights exp(lse_i - lse).
      const long prow = (long)blockIdx.z * ((long)a.B * a.K * a.G * a.T) + row;
      float* dst = a.part_o + prow * H;
#pragma unroll 1
      for (int c = 0; c < H; c += 32) {
        uint32_t ov[32];
        if (have) {
          tmem_ld32(tmem + lane_base + c, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0;
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst + c)[i] =
                make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                            __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
        }
      }
      if (valid) a.part_lse[prow] = lse_row;
    } else {
      stage_o_row<H>(sm + L::q_off, tmem, lane_base, 0, r, have, inv);
      if (valid) a.lse[row] = lse_row;
      fence_proxy_async_smem();
      named_bar_sync(1, kRows);
      if (tid == 0) {
        for (int c = 0; c < HC; ++c)
          tma_store_4d(&a.tm_o, sbase + L::q_off + c * kChunkBytes, c * 64, t0, 0, bk);
        bulk_commit();
        bulk_wait_read0();
      }
    }
  }

  // The Q copy started at entry must have landed before the CTA exits (it
  // has unless this CTA had no tiles or gave up waiting).
  if (tid == 0) mbar_wait_teardown(bars.q_full(), 0, a.wait_limit_ns);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Persistent forward for H <= 128 without split-KV.  One CTA per SM walks the
// LPT-ordered Q tiles (items) blockIdx.x, blockIdx.x + gridDim.x, ...  The Q
// tile and the O accumulator of an item are double buffered (b = local item
// index & 1) and its KV-tile schedule sits in a ring of kSchedBufs lists, so a
// scheduler warp classifies the KV tiles of items ahead and starts the next Q
// copy while item k runs, the MMA warps compute the first S tiles of item k+1
// before item k is done, and the softmax warps run item k's epilogue after the
// first tile of item k+1.  Roles (256 threads): warps 0-3 softmax and epilogue, warp 4
// K/V producer, warp 5 S = Q K^T issuer and TMEM owner, warp 6 scheduler,
// warp 7 O += P V issuer.  One thread issuing both products is the limit at
// H <= 128 (a trace: ~87 cycles per S product and ~123 per P V product against
// 64 on the tensor pipe), so each product type has its own issuing warp.
// Tensor memory: O[b] at columns [128 b, 128 b + H), S buffers at 256 and 384.
constexpr int kPThreads = 256;
constexpr int kSchedBufs = 4;  // KV-tile schedules in flight (items)

template <int H>
struct PFwdSmem {
  static constexpr int HC = H / 64;
  static constexpr uint32_t q_off = 0;  // Q[b] at q_off + b * HC * kChunkBytes
  static constexpr uint32_t ring_off = 2 * HC * kChunkBytes;
  static constexpr uint32_t sched_off = ring_off + kSlots * kChunkBytes;  // uint16[kSchedBufs][kMaxKvTiles]
  static constexpr uint32_t runs_off = sched_off + kSchedBufs * kMaxKvTiles * 2;  // uint8[kSchedBufs][kMaxKvTiles]
  static constexpr uint32_t bar_off = runs_off + kSchedBufs * kMaxKvTiles;
  // q_full[2], item_free[2], sched_full[kSchedBufs], list_free[kSchedBufs], then
  // the Bars block (full, empty, s_full, p_full, pv_done, teardown), the
  // O += P V issuer's teardown, and o_staged
  static constexpr int n_head = 4 + 2 * kSchedBufs;
  static constexpr int n_bars = n_head + 1 + 2 * kSlots + 7 + 1 + 1;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;  // tmem slot, abort, item info[kSchedBufs][4]
  static constexpr uint32_t bytes = misc_off + 16 + kSchedBufs * 16;
  static constexpr uint32_t alloc = bytes + 1024;
};

template <int H>
__global__ void __launch_bounds__(kPThreads, 1) fa_fwd_persistent_kernel(const __grid_constant__ FwdArgs a) {
  using L = PFwdSmem<H>;
  constexpr int HC = L::HC;
  constexpr int CC = fwd_copy_chunks(H);  // chunks per K/V copy
  static_assert(H <= 128, "two O accumulators must fit next to the S buffers");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t pb = sbase + L::bar_off;
  // Q[b] and O[b] are double buffered by item (b = k & 1); the KV-tile
  // schedule of item k sits in list buffer k % kSchedBufs, so the scheduler
  // classifies up to kSchedBufs - 2 items ahead of the Q buffers' release.
  auto q_full = [&](int b) { return pb + 8 * b; };
  auto item_free = [&](int b) { return pb + 8 * (2 + b); };
  auto sched_full = [&](int sb) { return pb + 8 * (4 + sb); };
  auto list_free = [&](int sb) { return pb + 8 * (4 + kSchedBufs + sb); };
  Bars bars{pb + 8 * L::n_head};
  const uint32_t teardown_pv = pb + 8 * (L::n_head + 1 + 2 * kSlots + 7);
  // every softmax thread has staged its row of O / l: the storing thread waits
  // on it with a bound (a named barrier could not give up if a warp aborted
  // before reaching it)
  const uint32_t o_staged = pb + 8 * (L::n_head + 1 + 2 * kSlots + 7 + 1);
  auto sched = [&](int b) { return reinterpret_cast<uint16_t*>(sm + L::sched_off) + b * kMaxKvTiles; };
  // segment-run byte of each schedule entry (segment ids only)
  auto runs_of = [&](int b) { return sm + L::runs_off + b * kMaxKvTiles; };
  auto q_tile = [&](int b) { return L::q_off + (uint32_t)b * HC * kChunkBytes; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc_off + 4);
  volatile int* info_all = reinterpret_cast<volatile int*>(sm + L::misc_off + 16);  // [kSchedBufs][4]
  const Abort ab{abort_flag, a.wait_limit_ns, a.err};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tb = kRows / a.G;
  const int BKn = a.B * a.K;
  const int n_items = a.n_qtiles * BKn;
  const int off = a.S - a.T;
  const int n_kv_all = (a.S + kKvRows - 1) / kKvRows;
  const bool segs = a.seg_q != nullptr;

  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full(b), 1);
      // producer done with the item, both MMA warps have read the tile count,
      // epilogue stored: Q[b] and O[b] may be refilled
      mbar_init(item_free(b), 4);
    }
    for (int sb = 0; sb < kSchedBufs; ++sb) {
      mbar_init(sched_full(sb), 1);
      // the producer and the four softmax warps have read the item's list
      mbar_init(list_free(sb), 5);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full(i), 1);
      mbar_init(bars.p_full(i), kRows);
      mbar_init(bars.pv_done(i), 1);
    }
    mbar_init(bars.teardown(), 1);
    mbar_init(teardown_pv, 1);
    mbar_init(o_staged, kRows);
    fence_barrier_init();
  }
  if (warp == 5) { tmem_alloc(smem_u32(tmem_slot), 512); tmem_relinquish(); }
  if (warp == 4) { prefetch_tmap(&a.tm_k); prefetch_tmap(&a.tm_v); }
  if (warp == 6) { prefetch_tmap(&a.tm_q); prefetch_tmap(&a.tm_o); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 6) {
    // ---------------------------------------------------------- scheduler
    bool ok = true;
    int k = 0;
    for (;; ++k) {
      const int b = k & 1, sb = k % kSchedBufs;
      // list buffer sb was last read by item k - kSchedBufs
      if (k >= kSchedBufs && !warp_wait(list_free(sb), ((k / kSchedBufs) - 1) & 1, ab)) { ok = false; break; }
      volatile int* info = info_all + 4 * sb;
      // Snake order over the LPT list: even rounds left to right, odd rounds
      // right to left, so every CTA's share of the decreasing sizes evens out.
      const int G = (int)gridDim.x;
      const int item = k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
      if (item >= n_items) {
        if (lane == 0) { info[0] = -1; mbar_arrive(sched_full(sb)); }
        break;
      }
      const int qt = a.n_qtiles - 1 - item / BKn, bk = item % BKn, bb = bk / a.K;
      const int t0 = qt * Tb, n_valid = min(Tb, a.T - t0);
      int n_kv = n_kv_all;
      if (a.causal) {
        const int lim = t0 + n_valid - 1 + off;
        n_kv = lim < 0 ? 0 : min(n_kv_all, lim / kKvRows + 1);
      }
      int qmn = INT_MAX, qmx = INT_MIN;
      if (segs) {
        for (int i = lane; i < n_valid; i += 32) {
          const int v = a.seg_q[(long)bb * a.T + t0 + i];
          qmn = min(qmn, v);
          qmx = max(qmx, v);
        }
        qmn = __reduce_min_sync(0xffffffffu, qmn);
        qmx = __reduce_max_sync(0xffffffffu, qmx);
      }
      // Classify 32 KV tiles at a time, one per lane, and compact the
      // non-empty ones (ballot prefix sums) into the schedule.
      uint16_t* list = sched(sb);
      int count = 0;
      for (int j0 = 0; j0 < n_kv; j0 += 32) {
        const int j = j0 + lane;
        uint8_t c = TILE_EMPTY, run = kRunsGeneral;
        if (j < n_kv) {
          c = TILE_FULL;
          const int s_first = j * kKvRows, s_last = min(s_first + kKvRows, a.S) - 1;
          if (a.causal && s_last > t0 + off) c = TILE_PARTIAL;  // crosses the diagonal
          if (s_first + kKvRows > a.S) c = TILE_PARTIAL;         // ragged last tile
          if (segs) {
            int mn = INT_MAX, mx = INT_MIN;
            // where the id changes, if it changes at most once
            int prev = 0, changes = 0, pos = kKvRows;
            const int32_t* ids = a.seg_kv + (long)bb * a.S + s_first;
            if ((a.S & 3) == 0 && s_first + kKvRows <= a.S) {
              const int4* kid = reinterpret_cast<const int4*>(ids);
#pragma unroll 8
              for (int e = 0; e < kKvRows / 4; ++e) {
                const int4 v = __ldg(kid + e);
                mn = min(min(mn, v.x), min(v.y, min(v.z, v.w)));
                mx = max(max(mx, v.x), max(v.y, max(v.z, v.w)));
                if (e > 0 && v.x != prev && changes++ == 0) pos = 4 * e;
                if (v.y != v.x && changes++ == 0) pos = 4 * e + 1;
                if (v.z != v.y && changes++ == 0) pos = 4 * e + 2;
                if (v.w != v.z && changes++ == 0) pos = 4 * e + 3;
                prev = v.w;
              }
            } else {
              for (int e = 0; e <= s_last - s_first; ++e) {
                const int v = __ldg(ids + e);
                mn = min(mn, v);
                mx = max(mx, v);
                if (e > 0 && v != prev && changes++ == 0) pos = e;
                prev = v;
              }
            }
            if (mx < qmn || mn > qmx) c = TILE_EMPTY;
            else if (!(mn == mx && qmn == qmx && mn == qmn)) c = TILE_PARTIAL;
            run = changes == 0 ? (uint8_t)kKvRows : changes == 1 ? (uint8_t)pos : kRunsGeneral;
          }
          if (c != TILE_EMPTY && a.bm.cls != nullptr)  // the Q tile lies inside one 128-position block
            c = (uint8_t)class_and(c, bm_tile_class(a.bm, bk % a.K, a.G, t0 >> 7, j));
        }
        const uint32_t m = __ballot_sync(0xffffffffu, c != TILE_EMPTY);
        if (c != TILE_EMPTY) {
          const int at = count + __popc(m & ((1u << lane) - 1));
          list[at] = (uint16_t)(j | (c == TILE_PARTIAL ? 0x8000 : 0));
          runs_of(sb)[at] = run;
        }
        count += __popc(m);
      }
      __syncwarp();
      // Q[b] and O[b] were last used by item k - 2
      if (k >= 2 && !warp_wait(item_free(b), ((k >> 1) - 1) & 1, ab)) { ok = false; break; }
      if (lane == 0) {
        info[0] = count; info[1] = qt; info[2] = bk;
        if (count > 0) {
          mbar_arrive_expect_tx(q_full(b), HC * kChunkBytes);
          for (int c = 0; c < HC; ++c)
            tma_load_4d(sbase + q_tile(b) + c * kChunkBytes, &a.tm_q, q_full(b), c * 64, t0, 0, bk);
        } else {
          mbar_arrive(q_full(b));  // keep the phase count of q_full(b) in step
        }
        mbar_arrive(sched_full(sb));
      }
    }
    // Q copies still in flight (the last two items) land before the CTA exits.
    if (lane == 0) {
      for (int kk = max(0, k - 2); kk < k; ++kk)
        mbar_wait_teardown(q_full(kk & 1), (kk >> 1) & 1, a.wait_limit_ns);
    }
    (void)ok;
  } else if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t seq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int b = k & 1, sb = k % kSchedBufs;
        if (!mbar_wait(sched_full(sb), (k / kSchedBufs) & 1, ab)) { ok = false; break; }
        volatile int* info = info_all + 4 * sb;
        const int n_tiles = info[0];
        if (n_tiles < 0) break;
        const int bk = info[2];
        const uint16_t* list = sched(sb);
        for (int u = 0; u < 2 * n_tiles && ok; ++u) {
          // unit 0: K(0); last unit: V(N-1); odd u: K((u+1)/2); even u: V(u/2 - 1)
          bool is_k;
          int n;
          if (u == 0) { is_k = true; n = 0; }
          else if (u == 2 * n_tiles - 1) { is_k = false; n = n_tiles - 1; }
          else if (u & 1) { is_k = true; n = (u + 1) / 2; }
          else { is_k = false; n = u / 2 - 1; }
          const int j = list[n] & 0x7fff;
          const CUtensorMap* m = is_k ? &a.tm_k : &a.tm_v;
          // The unit's HC chunks sit in consecutive slots (kSlots is a multiple
          // of HC).  Each copy fills CC of them and completes on the first one's
          // barrier, once every chunk's previous reader has released its slot.
          for (int cc = 0; cc < HC && ok; cc += CC, seq += CC) {
            for (int c = 0; c < CC && ok; ++c) {
              const uint32_t sq = seq + c;
              if (sq >= kSlots && !mbar_wait(bars.empty(sq % kSlots), ((sq / kSlots) - 1) & 1, ab)) ok = false;
            }
            if (!ok) break;
            const int slot = seq % kSlots;
            mbar_arrive_expect_tx(bars.full(slot), CC * kChunkBytes);
            tma_load_4d(sbase + L::ring_off + slot * kChunkBytes, m, bars.full(slot), 0, j * kKvRows, cc, bk);
          }
        }
        if (ok) {  // done with this item's schedule
          mbar_arrive(list_free(sb));
          mbar_arrive(item_free(b));
        }
      }
      if (!ok) {
        const uint32_t first = seq > kSlots ? seq - kSlots : 0;
        for (uint32_t q = first; q < seq; q += CC)  // one copy per CC chunks, on its first slot
          mbar_wait_teardown(bars.full(q % kSlots), (q / kSlots) & 1, a.wait_limit_ns);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
      const uint64_t dk0 = sdesc_sw128(sbase + L::ring_off, 16, 1024);
      bool ok = true;
      uint32_t seq_base = 0;  // ring chunks of earlier items
      int N = 0;              // tiles of earlier items (S / P buffer and parity counter)
      for (int k = 0; ok; ++k) {
        const int b = k & 1, sb = k % kSchedBufs;
        if (!mbar_wait(sched_full(sb), (k / kSchedBufs) & 1, ab)) { ok = false; break; }
        const int n_tiles = info_all[4 * sb];
        if (n_tiles < 0) break;
        // Nothing else of the item's shared state is read here (Q[b] is
        // released by the epilogue, which waits for every product of the item).
        mbar_arrive(item_free(b));
        if (n_tiles == 0) continue;
        if (!mbar_wait(q_full(b), (k >> 1) & 1, ab)) { ok = false; break; }
        const uint64_t dq0 = sdesc_sw128(sbase + q_tile(b), 16, 1024);
        for (int n = 0; n < n_tiles && ok; ++n) {
          const int Nn = N + n;
          // S buffer Nn&1 holds P of tile Nn-2 until O += P V of that tile is done.
          if (Nn >= 2 && !mbar_wait(bars.pv_done(Nn & 1), ((Nn - 2) >> 1) & 1, ab)) { ok = false; break; }
          const uint32_t s_col = 256 + 128 * (Nn & 1);
          const uint32_t seq0 = seq_base + unit_k(n) * HC;
          const int slot0 = seq0 % kSlots;
          for (int c = 0; c < HC && ok; ++c) {
            if (!mbar_wait(bars.full(slot0 + c - c % CC), (seq0 / kSlots) & 1, ab)) { ok = false; break; }
            tc_fence_after();
            const uint64_t qa = sdesc_add(dq0, c * kChunkBytes);
            const uint64_t kb = sdesc_add(dk0, (slot0 + c) * kChunkBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + s_col, sdesc_add(qa, kk * 32), sdesc_add(kb, kk * 32), id_s,
                     (c > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bars.empty(slot0 + c));
          }
          if (!ok) break;
          mma_commit(bars.s_full(Nn & 1));
        }
        seq_base += 2u * n_tiles * HC;
        N += n_tiles;
      }
      if (!ok) {
        mma_commit(bars.teardown());
        mbar_wait_teardown(bars.teardown(), 0, a.wait_limit_ns);
      }
    }
  } else if (warp == 7) {
    // ------------------------------------------------------ O += P V issuer
    if (lane == 0) {
      constexpr uint32_t id_o = idesc_bf16(128, H, false, true);  // N = H, V MN-major
      const uint64_t dv0 = sdesc_sw128(sbase + L::ring_off, kChunkBytes, 1024);
      bool ok = true;
      uint32_t seq_base = 0;
      int N = 0;
      for (int k = 0; ok; ++k) {
        const int b = k & 1, sb = k % kSchedBufs;
        if (!mbar_wait(sched_full(sb), (k / kSchedBufs) & 1, ab)) { ok = false; break; }
        const int n_tiles = info_all[4 * sb];
        if (n_tiles < 0) break;
        mbar_arrive(item_free(b));
        const uint32_t o_col = 128u * b;  // free: sched_full follows item k-2's release of O[b]
        for (int n = 0; n < n_tiles && ok; ++n) {
          const int Nn = N + n;
          if (!mbar_wait(bars.p_full(Nn & 1), (Nn >> 1) & 1, ab)) { ok = false; break; }
          const uint32_t seq0 = seq_base + unit_v(n, n_tiles) * HC;
          const int slot0 = seq0 % kSlots;  // the unit's HC chunks sit in consecutive slots
          for (int c = 0; c < HC && ok; c += CC)  // every copy of the V tile
            if (!mbar_wait(bars.full(slot0 + c), (seq0 / kSlots) & 1, ab)) ok = false;
          if (!ok) break;
          tc_fence_after();
          const uint32_t p_col = 256 + 128 * (Nn & 1);
          const uint64_t bv = sdesc_add(dv0, slot0 * kChunkBytes);
#pragma unroll
          for (int kk = 0; kk < kKvRows / 16; ++kk)
            mma_ts(tmem + o_col, tmem + p_col + kk * 8, sdesc_add(bv, kk * 2048), id_o,
                   (n > 0 || kk > 0) ? 1u : 0u);
          for (int c = 0; c < HC; ++c) mma_commit(bars.empty(slot0 + c));
          mma_commit(bars.pv_done(Nn & 1));
        }
        seq_base += 2u * n_tiles * HC;
        N += n_tiles;
      }
      if (!ok) {
        mma_commit(teardown_pv);
        mbar_wait_teardown(teardown_pv, 0, a.wait_limit_ns);
      }
    }
  } else {
    // --------------------------------------------------- softmax, epilogue
    // The epilogue of item k runs after the first softmax tile of item k + 1,
    // so the tensor core has that tile's products to work on meanwhile (O is
    // double buffered per item).  Thread 0 awaits the read of a TMA store one
    // tile later, before it frees the item's buffers.
    const int r = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int g = r / Tb;
    bool ok = true;
    int N = 0;
    // the item whose epilogue is pending
    bool pend = false;
    int p_k = 0, p_tiles = 0, p_last = 0, p_t0 = 0, p_bk = 0;
    float p_m = -INFINITY, p_l = 0.f;
    int free_b = -1;  // thread 0: buffers whose O store still reads shared memory
    auto release = [&]() {
      if (tid == 0 && free_b >= 0) {
        bulk_wait_read0();
        mbar_arrive(item_free(free_b));  // Q[b] (staging) and O[b] may be reused
        free_b = -1;
      }
    };
    auto finish = [&]() -> bool {
      pend = false;
      const int b = p_k & 1;
      const bool have = p_tiles > 0 && warp_wait(bars.pv_done(p_last & 1), (p_last >> 1) & 1, ab);
      if (p_tiles > 0 && !have) return false;
      if (have) tc_fence_after();
      const float inv = (have && p_l > 0.f) ? 1.f / p_l : 0.f;
      const float lse_row = (have && p_l > 0.f) ? (p_m + __log2f(p_l)) * kLn2 : -INFINITY;
      // Q[b] is free: every product of the item has completed (pv_done of its
      // last tile follows them all), or there were none.
      stage_o_row<H>(sm + q_tile(b), tmem, lane_base, 128u * b, r, have, inv);
      const int t = p_t0 + (r - g * Tb);
      if (t < a.T) a.lse[((long)p_bk * a.G + g) * a.T + t] = lse_row;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(o_staged);
      bool stored = true;
      if (warp == 0) {  // the outcome of thread 0's wait is the whole warp's
        if (lane == 0) {
          release();
          stored = mbar_wait(o_staged, p_k & 1, ab);
          if (stored) {
            for (int c = 0; c < HC; ++c)
              tma_store_4d(&a.tm_o, sbase + q_tile(b) + c * kChunkBytes, c * 64, p_t0, 0, p_bk);
            bulk_commit();
            free_b = b;
          }
        }
        stored = __shfl_sync(0xffffffffu, stored, 0);
      }
      return stored;
    };
    for (int k = 0; ok; ++k) {
      const int b = k & 1, sb = k % kSchedBufs;
      release();  // the scheduler waits for it before it refills buffers b
      if (!warp_wait(sched_full(sb), (k / kSchedBufs) & 1, ab)) { ok = false; break; }
      volatile int* info = info_all + 4 * sb;
      const int n_tiles = info[0];
      if (n_tiles < 0) break;
      const int qt = info[1], bk = info[2], bb = bk / a.K;
      const int t0 = qt * Tb, t = t0 + (r - g * Tb);
      const bool valid = t < a.T;
      const int my_seg = (segs && valid) ? a.seg_q[(long)bb * a.T + t] : 0;
      const uint16_t* list = sched(sb);
      const uint8_t* runs = runs_of(sb);
      const uint32_t o_col = 128u * b;
      float m_ref = -INFINITY, l = 0.f;
      for (int n = 0; n < n_tiles; ++n) {
        if (!softmax_tile<H>(a, tmem, lane_base, list[n], runs[n], n, N + n, t, g, valid, my_seg, bb,
                             bk % a.K, bars, ab, m_ref, l, o_col)) {
          ok = false;
          break;
        }
        if (n == 0 && pend) {
          if (!finish()) { ok = false; break; }
        } else {
          release();
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(list_free(sb));  // this warp has read the item's list
      if (pend && !finish()) { ok = false; break; }  // an item without tiles
      pend = true;
      p_k = k; p_tiles = n_tiles; p_last = N + n_tiles - 1; p_t0 = t0; p_bk = bk;
      p_m = m_ref; p_l = l;
      N += n_tiles;
    }
    if (ok && pend) ok = finish();
    release();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void fill_empty_kernel(__nv_bfloat16* o, float* lse, long rows, int H) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < rows * H) o[i] = __float2bfloat16(0.f);
  if (i < rows) lse[i] = -INFINITY;
}

__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  const Abort ab{&flag, limit_ns, err};
  // Nothing ever arrives on this barrier: the bounded wait must give up.
  mbar_wait(smem_u32(&bar), 0, ab);
  __syncthreads();
}

template <int H>
cudaError_t launch_fwd_h(const FwdArgs& a, cudaStream_t st) {
  using L = FwdSmem<H>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<H>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(a.n_qtiles * a.B * a.K, 1, a.n_splits);
  fa_fwd_kernel<H><<<grid, kThreads, L::alloc, st>>>(a);
  return cudaGetLastError();
}

template <int H>
cudaError_t launch_fwd_persistent_h(const FwdArgs& a, int sm_count, cudaStream_t st) {
  using L = PFwdSmem<H>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_persistent_kernel<H>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const long items = (long)a.n_qtiles * a.B * a.K;
  const int grid = (int)(items < sm_count ? items : sm_count);
  fa_fwd_persistent_kernel<H><<<grid, kPThreads, L::alloc, st>>>(a);
  return cudaGetLastError();
}

// Merge split-KV partial results: one warp per query row.
//   lse = log sum_i exp(lse_i),  o = sum_i exp(lse_i - lse) * o_i
template <int H>
__global__ void split_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                     int n_splits, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                     long rows) {
  const long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int i = 0; i < n_splits; ++i) m = fmaxf(m, __ldg(part_lse + (long)i * rows + row));
  constexpr int PER = H / 32;  // columns per lane
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int i = 0; i < n_splits; ++i) {
      const float li = __ldg(part_lse + (long)i * rows + row);
      if (li == -INFINITY) continue;
      const float w = __expf(li - m);
      sum += w;
      const float* src = part_o + ((long)i * rows + row) * H + lane * PER;
#pragma unroll
      for (int j = 0; j < PER; j += 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src + j));
        acc[j] = fmaf(w, v.x, acc[j]);
        acc[j + 1] = fmaf(w, v.y, acc[j + 1]);
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16* dst = o + row * H + lane * PER;
#pragma unroll
  for (int j = 0; j < PER; j += 2)
    *reinterpret_cast<uint32_t*>(dst + j) = pack_bf16x2(acc[j] * inv, acc[j + 1] * inv);
  if (lane == 0) lse[row] = sum > 0.f ? m + __logf(sum) : -INFINITY;
}

}  // namespace

cudaError_t launch_split_combine(const float* part_o, const float* part_lse, int n_splits, void* o,
                                 float* lse, long rows, int H, cudaStream_t st) {
  const int warps = 8;
  const unsigned blocks = (unsigned)((rows + warps - 1) / warps);
  auto* ob = reinterpret_cast<__nv_bfloat16*>(o);
  switch (H) {
    case 64: split_combine_kernel<64><<<blocks, warps * 32, 0, st>>>(part_o, part_lse, n_splits, ob, lse, rows); break;
    case 128: split_combine_kernel<128><<<blocks, warps * 32, 0, st>>>(part_o, part_lse, n_splits, ob, lse, rows); break;
    case 256: split_combine_kernel<256><<<blocks, warps * 32, 0, st>>>(part_o, part_lse, n_splits, ob, lse, rows); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st, int schedule) {
  // schedule: 0 chooses (persistent for H <= 128 without split-KV when there
  // are more Q tiles than SMs: with one tile per CTA there is nothing to
  // overlap), 1 one CTA per Q tile, 2 persistent where supported.
  static int cached_dev = -1, cached_sms = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return cudaErrorInvalidValue;
    cached_sms = n;
    cached_dev = dev;
  }
  const int sms = cached_sms;
  const long items = (long)a.n_qtiles * a.B * a.K;
  const bool supported = a.H <= 128 && a.n_splits == 1;
  const bool persistent = supported && (schedule == 2 || (schedule == 0 && items > sms));
  switch (a.H) {
    case 64: return persistent ? launch_fwd_persistent_h<64>(a, sms, st) : launch_fwd_h<64>(a, st);
    case 128: return persistent ? launch_fwd_persistent_h<128>(a, sms, st) : launch_fwd_h<128>(a, st);
    case 256: return launch_fwd_h<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fill_empty(void* o, float* lse, long rows, int H, cudaStream_t st) {
  const long n = rows * (long)H > rows ? rows * (long)H : rows;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const long blocks = (n + threads - 1) / threads;
  fill_empty_kernel<<<(unsigned)blocks, threads, 0, st>>>(reinterpret_cast<__nv_bfloat16*>(o), lse,
                                                          rows, H);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa
