// Backward pass of blocked GQA flash attention on sm_103a.
//
// The pages give no backward; this is the derivative of the forward written
// out (P = exp(L - lse), dP = dO V^T, dS = P (dP - D), dq = dS K,
// dk = sum_g dS^T q, dv = sum_g P^T dO) in four launches:
//   1. preprocess   D[row] = sum_h dO * o (fp32), H / 8 lanes per row
//   2. seg ranges   per-tile [min, max] segment ids (only with SegmentIds)
//   3. dK/dV        one CTA per (kv tile, b*K): K and V stay in shared memory,
//                   the non-empty Q tiles (G heads packed, 128 rows) stream by;
//                   S = Q K^T and dP = dO V^T recomputed in TMEM, P and dS
//                   written to shared memory, and dV^T += dO^T P,
//                   dK^T += Q^T dS accumulated in TMEM with the head dim on the
//                   128 lanes (so H = 256 fits in tensor memory).  Where that
//                   grid is smaller than the GPU, up to 4 CTAs share a KV
//                   tile's Q tiles and the last to finish adds their fp32
//                   partial sums in a fixed order.
//   4. dQ           one CTA per (Q tile, b*K): Q and dO stay in shared memory,
//                   the non-empty KV tiles stream by; dS goes to TMEM as the A
//                   operand of dQ += dS K.
// The two gradient passes recompute S and dP (7 tile products instead of 5)
// and in exchange need no atomic accumulation: every output element is
// written once, by one CTA, from sums taken in a fixed order, so the result
// is deterministic.
#include <algorithm>
#include <cuda_bf16.h>
#include "block_mask.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

// dK/dV: warps 0-3 and 7-10 softmax side (two per TMEM lane quadrant, one per
// half of the key columns), 4 producer, 5-6 MMA issuers.
constexpr int kThreads = 352;
// dQ: warps 0-3 and 8-11 softmax side (two per TMEM lane quadrant, one per half
// of the key columns), 4 K producer, 5-6 MMA issuers, 7 V producer.
constexpr int kDqThreads = 384;
constexpr uint32_t kQChunk = 128 * 128;  // [128 rows x 64 dims] bf16
constexpr float kLog2e = 1.4426950408889634f;
enum : int { TILE_EMPTY = 0, TILE_FULL = 1, TILE_PARTIAL = 2 };

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  const bool ok = mbar_wait(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// Mask class of the (Q tile, KV tile) pair; the q tile covers positions
// [t0, min(t0 + Tb, T)), the kv tile [s0, min(s0 + kvr, S)).  Causal keeps
// s <= t + (S - T).  Segment ranges come from the per-tile [min, max] table
// (conservative for non-monotone ids).  Keys past S on a ragged last tile
// make it PARTIAL; query rows past T are handled by their -inf lse instead.
__device__ __forceinline__ int tile_class(const BwdArgs& a, const int2* qr, const int2* kr, int b,
                                          int kh, int qt, int jt, int Tb, int kvr) {
  const int t0 = qt * Tb, s0 = jt * kvr;
  const int t_last = min(t0 + Tb, a.T) - 1, s_last = min(s0 + kvr, a.S) - 1;
  const int off = a.S - a.T;
  int c = TILE_FULL;
  if (a.causal) {
    if (t_last + off < s0) return TILE_EMPTY;
    if (t0 + off < s_last) c = TILE_PARTIAL;
  }
  if (s0 + kvr > a.S) c = TILE_PARTIAL;
  if (a.seg_q != nullptr) {
    const int2 q = qr[(long)b * a.n_qtiles + qt];
    const int2 k = kr[(long)b * a.n_kvtiles + jt];
    if (k.y < q.x || k.x > q.y) return TILE_EMPTY;
    if (!(q.x == q.y && k.x == k.y && q.x == k.x)) c = TILE_PARTIAL;
  }
  if (a.bm.cls != nullptr)  // the Q tile lies in one mask block; kv tiles of <= 128 keys too
    c = class_and(c, bm_tile_class(a.bm, kh, a.G, t0 >> 7, s0 >> 7));
  return c;
}

// First Q tile a KV tile starting at s0 can see under the causal mask.
__device__ __forceinline__ int causal_first_qtile(const BwdArgs& a, int s0, int Tb) {
  if (!a.causal) return 0;
  const int x = s0 - (a.S - a.T) - Tb + 1;  // need qt*Tb + Tb - 1 + (S - T) >= s0
  return x <= 0 ? 0 : (x + Tb - 1) / Tb;
}

// One past the last KV tile (of kvr keys) the causal mask lets the rows
// [t0, min(t0 + Tb, T)) see.
__device__ __forceinline__ int causal_kv_end(const BwdArgs& a, int t0, int Tb, int kvr) {
  if (!a.causal) return a.n_kvtiles;
  const int lim = min(t0 + Tb, a.T) - 1 + (a.S - a.T);
  return lim < 0 ? 0 : min(a.n_kvtiles, lim / kvr + 1);
}

// The keys of a KV tile that a query row keeps, as far as the causal limit,
// the end of the keys and (for tiles whose segment ids form at most two runs)
// the row's segment id decide them: [klo, khi) relative to the tile's first
// key s0.  per_key: the tile's ids form more runs; mask32 then compares them
// one by one.
struct RowKeep {
  int klo, khi;
  bool per_key;
};
__device__ __forceinline__ RowKeep row_keep(const BwdArgs& a, int b, int jt, int s0, int t, int my_seg) {
  const int n_keys = min(a.kv_rows, a.S - s0);
  RowKeep k{0, n_keys, false};
  if (a.causal) k.khi = min(k.khi, t + (a.S - a.T) - s0 + 1);
  if (a.seg_q != nullptr) {
    const int runs = a.seg_runs[(long)b * a.n_kvtiles + jt];
    if (runs == kRunsGeneral) {
      k.per_key = true;
    } else {
      const int32_t* ids = a.seg_kv + (long)b * a.S + s0;
      if (my_seg == __ldg(ids)) k.khi = min(k.khi, runs);
      else if (runs < n_keys && my_seg == __ldg(ids + n_keys - 1)) k.klo = runs;
      else k.khi = 0;
    }
  }
  return k;
}

// Apply the mask to 32 consecutive key columns [scol, scol + 32) of the row at
// position t.  SEGS (segment ids given): `keep` is the row's row_keep for the
// tile starting at s0.  Without segment ids only the causal limit and the end
// of the keys apply, as one range of kept columns (and the block mask, as in
// both cases); those kernels carry no segment code at all.
template <bool SEGS>
__device__ __forceinline__ void mask32(float (&s)[32], const BwdArgs& a, int b, int kh, int g, int t,
                                       int my_seg, int scol, int s0, const RowKeep& keep) {
  if constexpr (SEGS) {
    const uint32_t kept = range_bits(keep.klo - (scol - s0), keep.khi - (scol - s0));
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!((kept >> i) & 1u)) s[i] = -INFINITY;
    if (keep.per_key) {
      const int32_t* ids = a.seg_kv + (long)b * a.S + scol;
      if ((a.S & 3) == 0 && scol + 32 <= a.S) {  // 16-byte aligned, in range: vector loads
        const int4* kid = reinterpret_cast<const int4*>(ids);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const int4 v = __ldg(kid + i4);
          if (v.x != my_seg) s[4 * i4 + 0] = -INFINITY;
          if (v.y != my_seg) s[4 * i4 + 1] = -INFINITY;
          if (v.z != my_seg) s[4 * i4 + 2] = -INFINITY;
          if (v.w != my_seg) s[4 * i4 + 3] = -INFINITY;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (scol + i < a.S && __ldg(ids + i) != my_seg) s[i] = -INFINITY;
      }
    }
  } else {
    int khi = a.S - scol;
    if (a.causal) khi = min(khi, t + (a.S - a.T) - scol + 1);
    const uint32_t kept = range_bits(0, khi);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!((kept >> i) & 1u)) s[i] = -INFINITY;
  }
  if (a.bm.cls != nullptr && t < a.T) {
    const uint32_t bits = bm_row_word(a.bm, kh, a.G, g, t, scol >> 7, (scol & 127) >> 5);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (!((bits >> i) & 1u)) s[i] = -INFINITY;
  }
}

// Row r, key columns [32c, 32c + 32) (16 bf16 pairs) into a [128 rows x BN keys]
// operand stored as [128 x 64] chunks with the 128-byte swizzle: 16-byte unit u
// of a row lands at unit u ^ (r % 8).
__device__ __forceinline__ void store_row32(uint8_t* base, int r, int c, const uint32_t* w) {
  const int chunk = (c * 32) / 64, u0 = ((c * 32) % 64) / 8;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t off = chunk * kQChunk + r * 128 + (((u0 + k) ^ (r & 7)) * 16);
    *reinterpret_cast<uint4*>(base + off) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}

// [lo, hi) covering every non-empty tile of a CTA's sweep, found by all
// threads at once (one class per thread and step, loads in parallel) so that
// the roles' loops skip the empty prefix and suffix of the sweep without one
// serial load per skipped tile.  Called by every thread (two __syncthreads);
// without segment ids or a block mask the classes need no loads.
template <typename ClassOf>
__device__ __forceinline__ int2 nonempty_range(int first, int end, int* lo_hi, ClassOf class_of) {
  if (threadIdx.x == 0) { lo_hi[0] = end; lo_hi[1] = first; }
  __syncthreads();
  int lo = end, hi = first;
  for (int x = first + (int)threadIdx.x; x < end; x += (int)blockDim.x)
    if (class_of(x) != TILE_EMPTY) { lo = min(lo, x); hi = max(hi, x + 1); }
  if (lo < end) atomicMin(lo_hi, lo);
  if (hi > first) atomicMax(lo_hi + 1, hi);
  __syncthreads();
  return make_int2(lo_hi[0], max(lo_hi[0], lo_hi[1]));
}

// Wait (whole warp) for the release barrier of every head-dim half.
template <int HH, typename F>
__device__ __forceinline__ bool wait_halves(F bar, uint32_t parity, const Abort& ab) {
#pragma unroll
  for (int h = 0; h < HH; ++h)
    if (!warp_wait(bar(h), parity, ab)) return false;
  return true;
}

// =================================================================== dQ
template <int H, int BN_>
struct DqCfg {
  static constexpr int BN = BN_;                       // keys per KV tile
  static constexpr int HC = H / 64;
  // TMEM buffers for S (dS overwrites it) and dP next to the H columns of dQ.
  // Two S buffers let S(n+1) run during the softmax of tile n; with H = 128,
  // BN = 128 only one dP buffer fits besides them (dQ 128 + S 2x128 + dP 128).
  static constexpr int NBS = (H + 3 * BN <= 512) ? 2 : 1;
  static constexpr int NBP = (H + NBS * BN + 2 * BN <= 512) ? 2 : 1;
  static_assert(H + (NBS + NBP) * BN <= 512, "tensor memory");
  static constexpr uint32_t KV_CHUNK = BN * 128;       // [BN rows x 64 dims]
  // K chunks live from S(n) to dQ(n), which trails S by NBS - 1 tiles; V chunks
  // from dP(n) only.  Separate rings keep the two lifetimes from blocking each
  // other.  H = 128 has room for a third K tile, so K(n+1) need not wait for
  // dQ(n-1).
  static constexpr int KSL = H == 256 ? 2 * HC : 3 * HC;
  static constexpr int VSL = H == 256 ? HC : 2 * HC;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t do_off = HC * kQChunk;
  static constexpr uint32_t k_off = 2 * HC * kQChunk;
  static constexpr uint32_t v_off = k_off + KSL * KV_CHUNK;
  static constexpr uint32_t bar_off = v_off + VSL * KV_CHUNK;
  // q_full, kfull[KSL], kempty[KSL], vfull[VSL], vempty[VSL], sdp_full[2], ds_full[2], dq_done[2], teardown[2]
  static constexpr int n_bars = 1 + 2 * KSL + 2 * VSL + 8;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t alloc = misc_off + 64 + 1024;
  static_assert(alloc <= 232448, "shared memory per CTA");
  __host__ __device__ static constexpr uint32_t s_col(int u) { return H + u * BN; }
  // Column (within an S buffer) of dS for keys [32 c, 32 c + 32): the keys of
  // each half of the tile are packed at the start of that half's S columns.
  __host__ __device__ static constexpr uint32_t ds_col(int c) {
    return (c / (BN / 64)) * (BN / 2) + (c % (BN / 64)) * 16;
  }
  __host__ __device__ static constexpr uint32_t dp_col(int u) { return H + NBS * BN + u * BN; }
};

template <int H, int BN_, bool SEGS>
__global__ void __launch_bounds__(kDqThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using C = DqCfg<H, BN_>;
  constexpr int HC = C::HC, BN = C::BN, NBS = C::NBS, NBP = C::NBP, KSL = C::KSL, VSL = C::VSL;
  // Hand-off barriers form a ring of two, tile n using entry n % 2 with parity (n / 2) & 1.
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + C::bar_off;
  auto q_full = [&] { return bar0; };
  auto kfull = [&](int s) { return bar0 + 8 * (1 + s); };
  auto kempty = [&](int s) { return bar0 + 8 * (1 + KSL + s); };
  auto vfull = [&](int s) { return bar0 + 8 * (1 + 2 * KSL + s); };
  auto vempty = [&](int s) { return bar0 + 8 * (1 + 2 * KSL + VSL + s); };
  constexpr int xb = 1 + 2 * KSL + 2 * VSL;
  auto sdp_full = [&](int u) { return bar0 + 8 * (xb + u); };
  auto ds_full = [&](int u) { return bar0 + 8 * (xb + 2 + u); };
  auto dq_done = [&](int u) { return bar0 + 8 * (xb + 4 + u); };
  auto teardown = [&](int i) { return bar0 + 8 * (xb + 6 + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::misc_off + 4);
  const Abort ab{abort_flag, a.wait_limit_ns, a.err};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tb = kRows / a.G;
  // Flat grid, Q-tile major: latest (causally heaviest) Q tiles of every head first.
  const int BKn = a.B * a.K;
  const int qt = a.n_qtiles - 1 - (int)(blockIdx.x / BKn);
  const int bk = (int)(blockIdx.x % BKn), b = bk / a.K;
  const int t0 = qt * Tb;
  const int2* qr = a.seg_ranges;  // read only when segment ids are given
  const int2* kr = qr + (long)a.B * a.n_qtiles;
  const int jt_end = causal_kv_end(a, t0, Tb, BN);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(q_full(), 1);
    for (int s = 0; s < KSL; ++s) { mbar_init(kfull(s), 1); mbar_init(kempty(s), 1); }
    for (int s = 0; s < VSL; ++s) { mbar_init(vfull(s), 1); mbar_init(vempty(s), 1); }
    for (int u = 0; u < 2; ++u) {
      mbar_init(sdp_full(u), 2);  // S (issuer A) and dP (issuer B)
      mbar_init(ds_full(u), 2 * kRows);
      mbar_init(dq_done(u), 1);
    }
    mbar_init(teardown(0), 1);
    mbar_init(teardown(1), 1);
    fence_barrier_init();
    // Q and dO at kernel entry: their latency overlaps set-up and classification
    mbar_arrive_expect_tx(q_full(), 2 * HC * kQChunk);
    for (int c = 0; c < HC; ++c) {
      tma_load_4d(sbase + C::q_off + c * kQChunk, &a.tm_q, q_full(), c * 64, t0, 0, bk);
      tma_load_4d(sbase + C::do_off + c * kQChunk, &a.tm_do, q_full(), c * 64, t0, 0, bk);
    }
  }
  if (warp == 5) { tmem_alloc(smem_u32(tmem_slot), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // (the loops start at 0 and skip [0, jr.x) with one compare: a loop start
  // read back from shared memory measured 15% slower at H = 256)
  const int2 jr = nonempty_range(0, jt_end, reinterpret_cast<int*>(sm + C::misc_off + 8), [&](int jt) {
    return tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN);
  });

  if (warp == 4) {
    // K producer (and the Q / dO tiles).  K chunks are held until dQ(n) is
    // done, V chunks only until dP(n): a separate V producer (warp 7) keeps
    // a V load from queueing behind a K slot that is still in use.
    if (lane == 0) {
      bool ok = true;
      uint32_t seq = 0;  // chunk sequence number
      uint32_t k_issued = 0;
      for (int jt = 0; jt < jr.y && ok; ++jt) {
        if (jt < jr.x || tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        for (int c = 0; c < HC && ok; ++c) {
          const uint32_t sq = seq + c;
          const int slot = sq % KSL;
          if (sq >= KSL && !mbar_wait(kempty(slot), ((sq / KSL) - 1) & 1, ab)) { ok = false; break; }
          mbar_arrive_expect_tx(kfull(slot), C::KV_CHUNK);
          tma_load_3d(sbase + C::k_off + slot * C::KV_CHUNK, &a.tm_k, kfull(slot), c * 64, jt * BN, bk);
          ++k_issued;
        }
        seq += HC;
      }
      if (!ok) {
        // Let copies in flight land before the CTA exits (bounded waits).
        for (uint32_t sq = k_issued > KSL ? k_issued - KSL : 0; sq < k_issued; ++sq)
          mbar_wait_teardown(kfull(sq % KSL), (sq / KSL) & 1, a.wait_limit_ns);
      }
    }
  } else if (warp == 7) {
    // V producer.
    if (lane == 0) {
      bool ok = true;
      uint32_t seq = 0, v_issued = 0;
      for (int jt = 0; jt < jr.y && ok; ++jt) {
        if (jt < jr.x || tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        for (int c = 0; c < HC && ok; ++c) {
          const uint32_t sq = seq + c;
          const int slot = sq % VSL;
          if (sq >= VSL && !mbar_wait(vempty(slot), ((sq / VSL) - 1) & 1, ab)) { ok = false; break; }
          mbar_arrive_expect_tx(vfull(slot), C::KV_CHUNK);
          tma_load_3d(sbase + C::v_off + slot * C::KV_CHUNK, &a.tm_v, vfull(slot), c * 64, jt * BN, bk);
          ++v_issued;
        }
        seq += HC;
      }
      if (!ok) {
        for (uint32_t sq = v_issued > VSL ? v_issued - VSL : 0; sq < v_issued; ++sq)
          mbar_wait_teardown(vfull(sq % VSL), (sq / VSL) & 1, a.wait_limit_ns);
      }
    }
  } else if (warp == 5) {
    // Issuer A: S = Q K^T and dQ += dS K (both read the K ring).
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, BN, false, false);
      constexpr uint32_t id_q = idesc_bf16(128, H, false, true);  // dQ += dS K, N = H
      const uint64_t dqd = sdesc_sw128(sbase + C::q_off, 16, 1024);
      const uint64_t dkk = sdesc_sw128(sbase + C::k_off, 16, 1024);                  // K, K-major
      const uint64_t dkm = sdesc_sw128(sbase + C::k_off, C::KV_CHUNK, 1024);         // K, MN-major
      bool ok = true, waited_q = false;
      int n = 0;
      // dQ(m) += dS(m) K(m); the HC chunks of K(m) sit in consecutive ring
      // slots, so one N = H product per 16 keys.
      auto issue_dq = [&](int m) -> bool {
        const int u = m % NBS;
        if (!mbar_wait(ds_full(m & 1), (m >> 1) & 1, ab)) return false;
        tc_fence_after();
        const int slot0 = (m * HC) % KSL;
        if constexpr (H == 256) {
          // Two N = 128 products, one per half of the head dims: the K chunks of
          // the first half are released while the second half still runs, so
          // the next K tile's first chunks (the ring holds only two tiles at
          // H = 256) start loading earlier.
          constexpr uint32_t id_h = idesc_bf16(128, 128, false, true);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint64_t bh = sdesc_add(dkm, (slot0 + 2 * hh) * C::KV_CHUNK);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts(tmem + hh * 128, tmem + C::s_col(u) + C::ds_col(kk / 2) + (kk & 1) * 8,
                     sdesc_add(bh, kk * 2048), id_h, (m > 0 || kk > 0) ? 1u : 0u);
            mma_commit(kempty(slot0 + 2 * hh));
            mma_commit(kempty(slot0 + 2 * hh + 1));
          }
        } else {
          const uint64_t b0 = sdesc_add(dkm, slot0 * C::KV_CHUNK);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem, tmem + C::s_col(u) + C::ds_col(kk / 2) + (kk & 1) * 8, sdesc_add(b0, kk * 2048),
                   id_q, (m > 0 || kk > 0) ? 1u : 0u);
          for (int c = 0; c < HC; ++c) mma_commit(kempty(slot0 + c));
        }
        mma_commit(dq_done(m & 1));
        return true;
      };
      for (int jt = 0; jt < jr.y && ok; ++jt) {
        if (jt < jr.x || tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        if (!waited_q) {
          if (!mbar_wait(q_full(), 0, ab)) { ok = false; break; }
          waited_q = true;
        }
        const int u = n % NBS;
        // S columns of buffer u held dS(n-NBS), read by dQ(n-NBS), which this
        // thread issued earlier (tcgen05.mma ops of one thread run in order).
        for (int c = 0; c < HC && ok; ++c) {
          const uint32_t sq = (uint32_t)n * HC + c;
          const int slot = sq % KSL;
          if (!mbar_wait(kfull(slot), (sq / KSL) & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t qa = sdesc_add(dqd, c * kQChunk), kb = sdesc_add(dkk, slot * C::KV_CHUNK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + C::s_col(u), sdesc_add(qa, kk * 32), sdesc_add(kb, kk * 32), id_s,
                   (c > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(sdp_full(n & 1));
        if (n >= NBS - 1 && !issue_dq(n - (NBS - 1))) { ok = false; break; }
        ++n;
      }
      for (int m = n - (NBS - 1); ok && m < n; ++m)
        if (m >= 0 && !issue_dq(m)) ok = false;
      if (!ok) {
        mma_commit(teardown(0));
        mbar_wait_teardown(teardown(0), 0, a.wait_limit_ns);
      }
    }
  } else if (warp == 6) {
    // Issuer B: dP = dO V^T.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, BN, false, false);
      const uint64_t ddo = sdesc_sw128(sbase + C::do_off, 16, 1024);
      const uint64_t dvk = sdesc_sw128(sbase + C::v_off, 16, 1024);
      bool ok = true, waited_q = false;
      int n = 0;
      for (int jt = 0; jt < jr.y && ok; ++jt) {
        if (jt < jr.x || tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        if (!waited_q) {
          if (!mbar_wait(q_full(), 0, ab)) { ok = false; break; }
          waited_q = true;
        }
        const int u = n % NBP;
        // dP columns of buffer u are free once the softmax side has read dP(n-NBP)
        // (it signals ds_full after reading).
        if (n >= NBP && !mbar_wait(ds_full((n - NBP) & 1), ((n - NBP) >> 1) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        for (int c = 0; c < HC && ok; ++c) {
          const uint32_t sq = (uint32_t)n * HC + c;
          const int slot = sq % VSL;
          if (!mbar_wait(vfull(slot), (sq / VSL) & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = sdesc_add(ddo, c * kQChunk), vb = sdesc_add(dvk, slot * C::KV_CHUNK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + C::dp_col(u), sdesc_add(da, kk * 32), sdesc_add(vb, kk * 32), id_s,
                   (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(vempty(slot));
        }
        if (!ok) break;
        mma_commit(sdp_full(n & 1));
        ++n;
      }
      if (!ok) {
        mma_commit(teardown(1));
        mbar_wait_teardown(teardown(1), 0, a.wait_limit_ns);
      }
    }
  } else {
    // softmax side: packed query row r sits in TMEM lane r; the two warps of a
    // lane quadrant split the key columns (and, in the epilogue, the head dims)
    const int quad = warp & 3, half = warp >= 8 ? 1 : 0;
    const int r = quad * 32 + lane, g = r / Tb, t = t0 + (r - g * Tb);
    const bool valid = t < a.T;  // rows past T (ragged last tile) are inert
    const long row = ((long)bk * a.G + g) * a.T + t;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float lse = valid ? a.lse[row] : -INFINITY;
    const float lse2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
    const float Dr = valid ? a.delta[row] : 0.f;
    const int my_seg = (a.seg_q && valid) ? a.seg_q[(long)b * a.T + t] : 0;
    bool ok = true;
    int n = 0;
    for (int jt = 0; jt < jr.y; ++jt) {
      if (jt < jr.x) continue;
      const int cls = tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN);
      if (cls == TILE_EMPTY) continue;
      const int us = n % NBS, up = n % NBP;
      RowKeep keep{};
      if constexpr (SEGS)
        if (cls == TILE_PARTIAL) keep = row_keep(a, b, jt, jt * BN, t, my_seg);
      if (!warp_wait(sdp_full(n & 1), (n >> 1) & 1, ab)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
        uint32_t sv[32], pv[32];
        tmem_ld32(tmem + lane_base + C::s_col(us) + c * 32, sv);
        tmem_ld32(tmem + lane_base + C::dp_col(up) + c * 32, pv);
        tmem_wait_ld();
        float* s = reinterpret_cast<float*>(sv);
        if (cls == TILE_PARTIAL)
          mask32<SEGS>(*reinterpret_cast<float(*)[32]>(s), a, b, bk % a.K, g, t, my_seg, jt * BN + c * 32,
                       jt * BN, keep);
        uint32_t ds[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(fmaf(s[2 * i], kLog2e, -lse2));
          const float p1 = fast_exp2(fmaf(s[2 * i + 1], kLog2e, -lse2));
          const float d0 = p0 * (__uint_as_float(pv[2 * i]) - Dr);
          const float d1 = p1 * (__uint_as_float(pv[2 * i + 1]) - Dr);
          ds[i] = pack_bf16x2(d0, d1);
        }
        // dS (bf16, 2 per column) overwrites S columns this warp has read: the
        // half's dS goes to the start of the half's own S columns (the other
        // warp of the quadrant is still reading its half).
        tmem_st16(tmem + lane_base + C::s_col(us) + C::ds_col(c), ds);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full(n & 1));
      ++n;
    }
    // dQ in bf16 is staged in the Q tile's shared memory (every MMA is done)
    // with the Q box's swizzled layout and written by TMA stores.
    const bool have = n > 0 && ok && warp_wait(dq_done((n - 1) & 1), ((n - 1) >> 1) & 1, ab);
    if (have) tc_fence_after();
    // The staging below overwrites the Q tile: with no product issued, nothing
    // has waited for its copy yet.
    if (n == 0) mbar_wait_teardown(q_full(), 0, a.wait_limit_ns);
#pragma unroll 1
    for (int c = half * (H / 2); c < (half + 1) * (H / 2); c += 32) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tmem + lane_base + c, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0;
      }
      uint4 pk[4];
      uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
      for (int i = 0; i < 16; ++i) pw[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      uint8_t* chunk = sm + C::q_off + (c / 64) * kQChunk;
      const uint32_t u0 = (c % 64) / 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(chunk + sw128_offset(r, u0 + i)) = pk[i];
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 2 * kRows);
    if (tid == 0) {
      for (int c = 0; c < HC; ++c)  // (H = 64 runs as 128: its zero upper chunk is not stored)
        if (c * 64 < a.H) tma_store_4d(&a.tm_dq, sbase + C::q_off + c * kQChunk, c * 64, t0, 0, bk);
      bulk_commit();
      bulk_wait_read0();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// ====================================================== dK/dV epilogue
// Run by the 8 softmax-side warps (256 threads) of a dK/dV CTA: TMEM lanes
// carry the head dim (thread r of a quadrant pair owns dims r and 128 + r),
// columns the keys (`half` selects this warp's half of them).  Without a split
// (one CTA per KV tile) dV, dK go straight to bf16.  With the Q range of each
// KV tile split over q_splits CTAs, each CTA stores its fp32 partial sums, and
// the last CTA of the tile to finish (one atomic count per tile; no CTA ever
// waits for another) adds the q_splits partials in split order and stores
// bf16, so the result does not depend on which CTA finishes last.
// have == false: this CTA contributes zeros.
template <int H, int BN, bool SPLIT>
__device__ __forceinline__ void dkdv_epilogue(const BwdArgs& a, uint32_t tmem_dv, uint32_t tmem_dk,
                                              int r, int half, bool have, int jt, int split, int bk,
                                              volatile int* last_flag) {
  constexpr int HH = H / 128;
  const int s0 = jt * BN;
  // a.H <= H: with H = 64 the kernel runs as H = 128 over zero-filled upper
  // dims, whose rows of dK^T / dV^T are zero and are not stored.
  const int Hs = a.H;
  __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(a.dv) + ((long)bk * a.S + s0) * Hs;
  __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(a.dk) + ((long)bk * a.S + s0) * Hs;
  if constexpr (!SPLIT) {
#pragma unroll 1
    for (int h = 0; h < HH; ++h) {
      const int hd = h * 128 + r;
      if (hd >= Hs) continue;
#pragma unroll 1
      for (int c = half * BN / 2; c < (half + 1) * BN / 2; c += 32) {
        uint32_t vv[32], kv[32];
        if (have) {
          tmem_ld32(tmem_dv + h * BN + c, vv);
          tmem_ld32(tmem_dk + h * BN + c, kv);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) { vv[k] = 0; kv[k] = 0; }
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (s0 + c + k < a.S) {  // keys past S (ragged last tile) are not stored
            dv[(long)(c + k) * Hs + hd] = __float2bfloat16(__uint_as_float(vv[k]));
            dk[(long)(c + k) * Hs + hd] = __float2bfloat16(__uint_as_float(kv[k]));
          }
        }
      }
    }
  } else {
    const int NS = a.q_splits;
    constexpr long kTile = (long)BN * H;  // floats of one partial dV (or dK) tile
    const long BKn = (long)a.B * a.K;
    auto part = [&](int p) { return a.dkv_part + (((long)jt * NS + p) * BKn + bk) * 2 * kTile; };
    float* mine = part(split);
#pragma unroll 1
    for (int h = 0; h < HH; ++h) {
      const int hd = h * 128 + r;
#pragma unroll 1
      for (int c = half * BN / 2; c < (half + 1) * BN / 2; c += 32) {
        uint32_t vv[32], kv[32];
        if (have) {
          tmem_ld32(tmem_dv + h * BN + c, vv);
          tmem_ld32(tmem_dk + h * BN + c, kv);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) { vv[k] = 0; kv[k] = 0; }
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          mine[(long)(c + k) * H + hd] = __uint_as_float(vv[k]);
          mine[kTile + (long)(c + k) * H + hd] = __uint_as_float(kv[k]);
        }
      }
    }
    __threadfence();  // this CTA's partial is visible before its count
    named_bar_sync(1, 2 * kRows);
    if (r == 0 && half == 0) {
      int* cnt = a.dkv_count + (long)jt * BKn + bk;
      const bool last = atomicAdd(cnt, 1) == NS - 1;
      if (last) atomicExch(cnt, 0);  // every CTA of the tile has counted: ready for the next call
      *last_flag = last ? 1 : 0;
    }
    named_bar_sync(1, 2 * kRows);
    if (*last_flag == 0) return;
    __threadfence();
    // 16 keys at a time: each partial's 32 values are loaded before any is
    // added, then added in split order.
#pragma unroll 1
    for (int h = 0; h < HH; ++h) {
      const int hd = h * 128 + r;
      if (hd >= Hs) continue;
#pragma unroll 1
      for (int c = half * BN / 2; c < (half + 1) * BN / 2; c += 16) {
        float sv[16], sk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) { sv[k] = 0.f; sk[k] = 0.f; }
#pragma unroll 1
        for (int p = 0; p < NS; ++p) {
          const float* src = part(p) + (long)c * H + hd;
          float lv[16], lk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            lv[k] = __ldcg(src + (long)k * H);
            lk[k] = __ldcg(src + kTile + (long)k * H);
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) { sv[k] += lv[k]; sk[k] += lk[k]; }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (s0 + c + k < a.S) {
            dv[(long)(c + k) * Hs + hd] = __float2bfloat16(sv[k]);
            dk[(long)(c + k) * Hs + hd] = __float2bfloat16(sk[k]);
          }
        }
      }
    }
  }
}

// The Q tiles [lo, hi) of KV tile jt's sweep that CTA `split` of q_splits takes:
// equal shares of the tiles from the first one the causal bound lets see the tile.
__device__ __forceinline__ int2 split_qrange(int qt_begin, int n_qtiles, int split, int n_splits) {
  const int len = max(0, n_qtiles - qt_begin);
  return make_int2(qt_begin + (int)((long)len * split / n_splits),
                   qt_begin + (int)((long)len * (split + 1) / n_splits));
}

// ================================================================ dK/dV
// One Q stage (H = 256: a second 64 KB Q tile does not fit next to K, V, dO, P
// and dS).  S(i+1) follows dK^T(i), which reads the only Q buffer.
template <int H, int BN_>
struct Dkv1Cfg {
  static constexpr int BN = BN_;              // keys per CTA
  static constexpr int HC = H / 64;
  static constexpr int HH = H / 128;          // 128-lane halves of the head dim
  static constexpr int PC = BN / 64;          // 64-key chunks of P / dS
  static constexpr uint32_t KV_CHUNK = BN * 128;
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t v_off = HC * KV_CHUNK;
  static constexpr uint32_t q_off = 2 * HC * KV_CHUNK;
  static constexpr uint32_t do_off = q_off + HC * kQChunk;
  static constexpr uint32_t p_off = do_off + HC * kQChunk;
  static constexpr uint32_t ds_off = p_off + PC * kQChunk;
  static constexpr uint32_t bar_off = ds_off + PC * kQChunk;
  // kv_full, s_full, dp_full, p_full, ds_full, teardown[2], q_full[HC], do_full[HC],
  // q_empty[HH], do_empty[HH]
  static constexpr uint32_t misc_off = bar_off + (7 + 2 * HC + 2 * HH) * 8;
  static constexpr uint32_t alloc = misc_off + 64 + 1024;
  static constexpr uint32_t dv_col = 0;
  static constexpr uint32_t dk_col = HH * BN;
  static constexpr uint32_t s_col = 2 * HH * BN;
  static constexpr uint32_t dp_col = 2 * HH * BN + BN;
};

template <int H, int BN_, bool SPLIT, bool SEGS>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dkdv1_kernel(const __grid_constant__ BwdArgs a) {
  using C = Dkv1Cfg<H, BN_>;
  constexpr int HC = C::HC, HH = C::HH, BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + C::bar_off;
  const uint32_t kv_full = bar0, s_full = bar0 + 8, dp_full = bar0 + 16;
  const uint32_t p_full = bar0 + 24, ds_full = bar0 + 32;
  auto teardown = [&](int i) { return bar0 + 8 * (5 + i); };
  auto q_full = [&](int c) { return bar0 + 8 * (7 + c); };
  auto do_full = [&](int c) { return bar0 + 8 * (7 + HC + c); };
  // Q (dO) 128-dim half h is released once dK^T (dV^T) of that half is done.
  auto q_empty = [&](int h) { return bar0 + 8 * (7 + 2 * HC + h); };
  auto do_empty = [&](int h) { return bar0 + 8 * (7 + 2 * HC + HH + h); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::misc_off + 4);
  const Abort ab{abort_flag, a.wait_limit_ns, a.err};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tb = kRows / a.G;
  // Flat grid.  Unsplit: head-major, early (causally heaviest) KV tiles of a
  // head first, so the CTAs that sweep one head's Q/dO tiles run together
  // (fewer Q/dO re-reads from DRAM than interleaving the heads: 1.28 -> 1.26
  // ms at T=8192).  With SPLIT (a grid smaller than the GPU) KV-tile major,
  // the q_splits CTAs of a KV tile splitting its Q range.
  const int BKn = a.B * a.K, NS = SPLIT ? a.q_splits : 1;
  const int jt = SPLIT ? (int)(blockIdx.x / (BKn * NS)) : (int)(blockIdx.x % a.n_kvtiles);
  const int split = SPLIT ? (int)(blockIdx.x / BKn) % NS : 0;
  const int bk = SPLIT ? (int)(blockIdx.x % BKn) : (int)(blockIdx.x / a.n_kvtiles), b = bk / a.K;
  // The dQ kernel reads nothing this kernel writes: let it be scheduled on SMs
  // this grid frees in its tail (it is launched with programmatic serialization).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s0 = jt * BN;
  const int2* qr = a.seg_ranges;  // read only when segment ids are given
  const int2* kr = qr + (long)a.B * a.n_qtiles;
  const int2 qsw = split_qrange(causal_first_qtile(a, s0, Tb), a.n_qtiles, split, NS);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    for (int h = 0; h < HH; ++h) { mbar_init(q_empty(h), 1); mbar_init(do_empty(h), 1); }
    mbar_init(s_full, 1);           // S done (issuer A's commit)
    mbar_init(dp_full, 1);          // dP done (issuer B's commit)
    mbar_init(p_full, 2 * kRows);   // P written (softmax side)
    mbar_init(ds_full, 2 * kRows);  // dS written (softmax side)
    mbar_init(teardown(0), 1);
    mbar_init(teardown(1), 1);
    for (int c = 0; c < HC; ++c) { mbar_init(q_full(c), 1); mbar_init(do_full(c), 1); }
    fence_barrier_init();
    // K and V at kernel entry: their latency overlaps set-up and classification
    mbar_arrive_expect_tx(kv_full, 2 * HC * C::KV_CHUNK);
    for (int c = 0; c < HC; ++c) {
      tma_load_3d(sbase + C::k_off + c * C::KV_CHUNK, &a.tm_k, kv_full, c * 64, s0, bk);
      tma_load_3d(sbase + C::v_off + c * C::KV_CHUNK, &a.tm_v, kv_full, c * 64, s0, bk);
    }
  }
  if (warp == 5) { tmem_alloc(smem_u32(tmem_slot), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int2 qrng = nonempty_range(qsw.x, qsw.y, reinterpret_cast<int*>(sm + C::misc_off + 8),
                                   [&](int qt) { return tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN); });

  if (warp == 4) {
    // Producer: K, V once; per Q tile, dO (released after dV^T) then Q
    // (released after dK^T), one barrier per 64-dim chunk.
    if (lane == 0) {
      bool ok = true;
      int i = 0;
      uint32_t issued = 0;  // chunks issued for the current tile (bit c: q, bit HC+c: dO)
      for (int qt = qrng.x; qt < qrng.y && ok; ++qt) {
        if (tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        issued = 0;
        for (int h = 0; h < HH && ok; ++h) {
          if (i > 0 && !mbar_wait(do_empty(h), (i - 1) & 1, ab)) { ok = false; break; }
          for (int c = 2 * h; c < 2 * h + 2; ++c) {
            mbar_arrive_expect_tx(do_full(c), kQChunk);
            tma_load_4d(sbase + C::do_off + c * kQChunk, &a.tm_do, do_full(c), c * 64, qt * Tb, 0, bk);
            issued |= 1u << (HC + c);
          }
          if (i > 0 && !mbar_wait(q_empty(h), (i - 1) & 1, ab)) { ok = false; break; }
          for (int c = 2 * h; c < 2 * h + 2; ++c) {
            mbar_arrive_expect_tx(q_full(c), kQChunk);
            tma_load_4d(sbase + C::q_off + c * kQChunk, &a.tm_q, q_full(c), c * 64, qt * Tb, 0, bk);
            issued |= 1u << c;
          }
        }
        if (!ok) break;
        ++i;
      }
      if (!ok) {
        // Let the copies of the tile being loaded land before the CTA exits.
        const int last = ok ? i - 1 : i;
        for (int c = 0; c < HC; ++c) {
          if (issued & (1u << c)) mbar_wait_teardown(q_full(c), last & 1, a.wait_limit_ns);
          if (issued & (1u << (HC + c))) mbar_wait_teardown(do_full(c), last & 1, a.wait_limit_ns);
        }
      }
    }
  } else if (warp == 5 || warp == 6) {
    // Two MMA issuers: A (warp 5) issues S = Q K^T and dK^T += Q^T dS (the Q
    // operand), B (warp 6) issues dP = dO V^T and dV^T += dO^T P (the dO operand).
    // P needs only S, so dV^T(i) starts while the softmax side still computes
    // dS(i) = P (dP - D); dK^T(i) follows once dS(i) is written.
    if (lane == 0) {
      const bool is_a = warp == 5;
      constexpr uint32_t id_s = idesc_bf16(128, BN, false, false);  // S, dP: [128 q x BN]
      constexpr uint32_t id_t = idesc_bf16(128, BN, true, true);    // dV^T, dK^T: [128 h x BN]
      const uint32_t x_off = is_a ? C::q_off : C::do_off;            // Q or dO tile
      const uint32_t y_off = is_a ? C::k_off : C::v_off;             // K or V tile
      const uint32_t z_off = is_a ? C::ds_off : C::p_off;            // dS or P
      const uint32_t d_col = is_a ? C::s_col : C::dp_col;            // S or dP
      const uint32_t acc_col = is_a ? C::dk_col : C::dv_col;         // dK^T or dV^T

      const uint64_t d_x = sdesc_sw128(sbase + x_off, 16, 1024);
      const uint64_t d_y = sdesc_sw128(sbase + y_off, 16, 1024);
      const uint64_t d_xT = sdesc_sw128(sbase + x_off, kQChunk, 1024);  // X^T, MN-major
      const uint64_t d_z = sdesc_sw128(sbase + z_off, kQChunk, 1024);
      bool ok = true;
      int i = 0;
      for (int qt = qrng.x; qt < qrng.y && ok; ++qt) {
        if (tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        if (i == 0 && !mbar_wait(kv_full, 0, ab)) { ok = false; break; }
        // S(i-1) was read before P(i-1) was signalled, and A waited for dS(i-1),
        // later still; dP(i-1) is read until dS(i-1) is signalled, so B waits here.
        if (!is_a && i > 0 && !mbar_wait(ds_full, (i - 1) & 1, ab)) { ok = false; break; }
        for (int c = 0; c < HC && ok; ++c) {
          if (!mbar_wait(is_a ? q_full(c) : do_full(c), i & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t xa = sdesc_add(d_x, c * kQChunk), yb = sdesc_add(d_y, c * C::KV_CHUNK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + d_col, sdesc_add(xa, kk * 32), sdesc_add(yb, kk * 32), id_s,
                   (c > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(is_a ? s_full : dp_full);
        if (!mbar_wait(is_a ? ds_full : p_full, i & 1, ab)) { ok = false; break; }
        tc_fence_after();
        for (int h = 0; h < HH; ++h) {  // contraction over the 128 packed query rows
          const uint64_t xA = sdesc_add(d_xT, 2 * h * kQChunk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + acc_col + h * BN, sdesc_add(xA, kk * 2048), sdesc_add(d_z, kk * 2048), id_t,
                   (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(is_a ? q_empty(h) : do_empty(h));  // this half of Q (dO) is free
        }
        ++i;
      }
      if (!ok) {
        mma_commit(teardown(is_a ? 0 : 1));
        mbar_wait_teardown(teardown(is_a ? 0 : 1), 0, a.wait_limit_ns);
      }
    }
  } else {
    // Softmax side: the row reads TMEM lane quadrant warp % 4; the two warps of
    // a quadrant split the key columns (no row reduction is needed: lse and D
    // are precomputed).
    const int quad = warp & 3, half = warp >= 7 ? 1 : 0;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    constexpr int NCH = BN / 64;  // 32-column chunks per warp
    bool ok = true;
    int i = 0;
    for (int qt = qrng.x; qt < qrng.y; ++qt) {
      const int cls = tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN);
      if (cls == TILE_EMPTY) continue;
      const int g = r / Tb, t = qt * Tb + (r - g * Tb);
      const bool valid = t < a.T;  // rows past T (ragged last tile) are inert
      const long row = ((long)bk * a.G + g) * a.T + t;
      const float lse = valid ? a.lse[row] : -INFINITY;
      const float lse2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
      const float Dr = valid ? a.delta[row] : 0.f;
      const int my_seg = (a.seg_q && valid) ? a.seg_q[(long)b * a.T + t] : 0;
      RowKeep keep{};
      if constexpr (SEGS)
        if (cls == TILE_PARTIAL) keep = row_keep(a, b, jt, s0, t, my_seg);
      // Phase 1: P = exp(S - lse) once S(i) is done.  s_full is A's commit, which
      // also covers dK^T(i-1) (the reader of the dS buffer); the P buffer's
      // reader dV^T(i-1) is B's, so its release barrier is waited for here.
      if (!warp_wait(s_full, i & 1, ab)) { ok = false; break; }
      if (i > 0 && !warp_wait(do_empty(HH - 1), (i - 1) & 1, ab)) { ok = false; break; }
      tc_fence_after();
      uint32_t pp[NCH][16];  // this warp's P (bf16 pairs), kept for phase 2
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = half * NCH + cc;
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + C::s_col + c * 32, sv);
        tmem_wait_ld();
        float* sf = reinterpret_cast<float*>(sv);
        if (cls == TILE_PARTIAL)
          mask32<SEGS>(*reinterpret_cast<float(*)[32]>(sf), a, b, bk % a.K, g, t, my_seg, s0 + c * 32, s0, keep);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pp[cc][k] = pack_bf16x2(fast_exp2(fmaf(sf[2 * k], kLog2e, -lse2)),
                                  fast_exp2(fmaf(sf[2 * k + 1], kLog2e, -lse2)));
        store_row32(sm + C::p_off, r, c, pp[cc]);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor cores
      tc_fence_before();
      mbar_arrive(p_full);
      // Phase 2: dS = P (dP - D) once dP(i) is done (masked entries have P = 0).
      if (!warp_wait(dp_full, i & 1, ab)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = half * NCH + cc;
        uint32_t pv[32], dd[16];
        tmem_ld32(tmem + lane_base + C::dp_col + c * 32, pv);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 pk = unpack_bf16x2(pp[cc][k]);
          dd[k] = pack_bf16x2(pk.x * (__uint_as_float(pv[2 * k]) - Dr),
                              pk.y * (__uint_as_float(pv[2 * k + 1]) - Dr));
        }
        store_row32(sm + C::ds_off, r, c, dd);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);
      ++i;
    }
    // Epilogue: lanes carry the head dim, columns the keys.
    const bool have = i > 0 && ok && warp_wait(q_empty(HH - 1), (i - 1) & 1, ab) &&
                      warp_wait(do_empty(HH - 1), (i - 1) & 1, ab);
    if (have) tc_fence_after();
    dkdv_epilogue<H, BN, SPLIT>(a, tmem + lane_base + C::dv_col, tmem + lane_base + C::dk_col, r, half,
                                have, jt, split, bk, reinterpret_cast<volatile int*>(sm + C::misc_off + 16));
  }
  if (tid == 0) mbar_wait_teardown(kv_full, 0, a.wait_limit_ns);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// ======================================================== dK/dV, two Q stages
// H = 128: the next Q tile has its own stage, so S(i+1) is issued as soon as the
// softmax side has read S(i) and the next tile's exponentials overlap this
// tile's dK^T / dV^T products.
template <int H, int BN_>
struct DkvCfg {
  static constexpr int BN = BN_;              // keys per CTA
  static constexpr int HC = H / 64;
  static constexpr int HH = H / 128;          // 128-lane halves of the head dim
  static constexpr int PC = BN / 64;          // 64-key chunks of P / dS
  // Q stages.  With H = 128 a second Q tile fits: S of the next Q tile is then
  // computed while the softmax side and dK^T / dV^T still work on this one.
  static constexpr int QB = 2;
  static_assert(H == 128, "two Q stages fit in shared memory at H = 128");
  static constexpr uint32_t KV_CHUNK = BN * 128;
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t v_off = HC * KV_CHUNK;
  static constexpr uint32_t q_off = 2 * HC * KV_CHUNK;  // QB stages of HC chunks
  static constexpr uint32_t do_off = q_off + QB * HC * kQChunk;
  static constexpr uint32_t p_off = do_off + HC * kQChunk;
  static constexpr uint32_t ds_off = p_off + PC * kQChunk;
  static constexpr uint32_t bar_off = ds_off + PC * kQChunk;
  // kv_full, s_full, dp_full, p_full, ds_full, teardown[2], q_full[QB][HC],
  // do_full[HC], q_empty[QB][HH], do_empty[HH]
  static constexpr int n_bars = 7 + QB * HC + HC + QB * HH + HH;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t alloc = misc_off + 64 + 1024;
  static_assert(alloc <= 232448, "shared memory per CTA");
  static constexpr uint32_t dv_col = 0;
  static constexpr uint32_t dk_col = HH * BN;
  static constexpr uint32_t s_col = 2 * HH * BN;
  static constexpr uint32_t dp_col = 2 * HH * BN + BN;
};

template <int H, int BN_, bool SPLIT, bool SEGS>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using C = DkvCfg<H, BN_>;
  constexpr int HC = C::HC, HH = C::HH, BN = C::BN, QB = C::QB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + C::bar_off;
  const uint32_t kv_full = bar0, s_full = bar0 + 8, dp_full = bar0 + 16;
  const uint32_t p_full = bar0 + 24, ds_full = bar0 + 32;
  auto teardown = [&](int i) { return bar0 + 8 * (5 + i); };
  // Tile i (i-th non-empty Q tile) uses Q stage i % QB, the (i / QB)-th use of it.
  auto q_full = [&](int qb, int c) { return bar0 + 8 * (7 + qb * HC + c); };
  auto do_full = [&](int c) { return bar0 + 8 * (7 + QB * HC + c); };
  // Q (dO) 128-dim half h is released once dK^T (dV^T) of that half is done.
  auto q_empty = [&](int qb, int h) { return bar0 + 8 * (7 + QB * HC + HC + qb * HH + h); };
  auto do_empty = [&](int h) { return bar0 + 8 * (7 + QB * HC + HC + QB * HH + h); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::misc_off + 4);
  const Abort ab{abort_flag, a.wait_limit_ns, a.err};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tb = kRows / a.G;
  // Flat grid, KV-tile major: early (causally heaviest) KV tiles of every head
  // first; with SPLIT the q_splits CTAs of a KV tile split its Q range.
  const int BKn = a.B * a.K, NS = SPLIT ? a.q_splits : 1;
  const int jt = (int)(blockIdx.x / (BKn * NS));
  const int split = SPLIT ? (int)(blockIdx.x / BKn) % NS : 0;
  const int bk = (int)(blockIdx.x % BKn), b = bk / a.K;
  // The dQ kernel reads nothing this kernel writes: let it be scheduled on SMs
  // this grid frees in its tail (it is launched with programmatic serialization).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s0 = jt * BN;
  const int2* qr = a.seg_ranges;  // read only when segment ids are given
  const int2* kr = qr + (long)a.B * a.n_qtiles;
  const int2 qsw = split_qrange(causal_first_qtile(a, s0, Tb), a.n_qtiles, split, NS);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    for (int h = 0; h < HH; ++h) {
      mbar_init(do_empty(h), 1);
      for (int qb = 0; qb < QB; ++qb) mbar_init(q_empty(qb, h), 1);
    }
    mbar_init(s_full, 1);           // S done (issuer A's commit)
    mbar_init(dp_full, 1);          // dP done (issuer B's commit)
    mbar_init(p_full, 2 * kRows);   // P written (softmax side)
    mbar_init(ds_full, 2 * kRows);  // dS written (softmax side)
    mbar_init(teardown(0), 1);
    mbar_init(teardown(1), 1);
    for (int c = 0; c < HC; ++c) {
      mbar_init(do_full(c), 1);
      for (int qb = 0; qb < QB; ++qb) mbar_init(q_full(qb, c), 1);
    }
    fence_barrier_init();
    // K and V at kernel entry: their latency overlaps set-up and classification
    mbar_arrive_expect_tx(kv_full, 2 * HC * C::KV_CHUNK);
    for (int c = 0; c < HC; ++c) {
      tma_load_3d(sbase + C::k_off + c * C::KV_CHUNK, &a.tm_k, kv_full, c * 64, s0, bk);
      tma_load_3d(sbase + C::v_off + c * C::KV_CHUNK, &a.tm_v, kv_full, c * 64, s0, bk);
    }
  }
  if (warp == 5) { tmem_alloc(smem_u32(tmem_slot), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int2 qrng = nonempty_range(qsw.x, qsw.y, reinterpret_cast<int*>(sm + C::misc_off + 8),
                                   [&](int qt) { return tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN); });

  if (warp == 4) {
    // Producer: K, V once; per Q tile, dO (released after dV^T) then Q
    // (released after dK^T), one barrier per 64-dim chunk.
    if (lane == 0) {
      bool ok = true;
      int i = 0;
      uint32_t issued = 0;  // chunks issued for the current tile (bit c: q, bit HC+c: dO)
      for (int qt = qrng.x; qt < qrng.y && ok; ++qt) {
        if (tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        issued = 0;
        const int qb = i % QB;
        auto load_q = [&](int h) -> bool {
          // stage qb was last read by dK^T of tile i - QB
          if (i >= QB && !mbar_wait(q_empty(qb, h), ((i / QB) - 1) & 1, ab)) return false;
          for (int c = 2 * h; c < 2 * h + 2; ++c) {
            mbar_arrive_expect_tx(q_full(qb, c), kQChunk);
            tma_load_4d(sbase + C::q_off + (qb * HC + c) * kQChunk, &a.tm_q, q_full(qb, c), c * 64,
                        qt * Tb, 0, bk);
            issued |= 1u << c;
          }
          return true;
        };
        auto load_do = [&](int h) -> bool {
          if (i > 0 && !mbar_wait(do_empty(h), (i - 1) & 1, ab)) return false;
          for (int c = 2 * h; c < 2 * h + 2; ++c) {
            mbar_arrive_expect_tx(do_full(c), kQChunk);
            tma_load_4d(sbase + C::do_off + c * kQChunk, &a.tm_do, do_full(c), c * 64, qt * Tb, 0, bk);
            issued |= 1u << (HC + c);
          }
          return true;
        };
        // Q first: its stage frees with dK^T of tile i - 2, long before dO's.
        for (int h = 0; h < HH && ok; ++h) ok = load_q(h);
        for (int h = 0; h < HH && ok; ++h) ok = load_do(h);
        if (!ok) break;
        ++i;
      }
      if (!ok) {
        // Let the copies of the tile being loaded land before the CTA exits.
        const int last = i;  // the tile being loaded when the producer gave up
        for (int c = 0; c < HC; ++c) {
          if (issued & (1u << c))
            mbar_wait_teardown(q_full(last % QB, c), (last / QB) & 1, a.wait_limit_ns);
          if (issued & (1u << (HC + c))) mbar_wait_teardown(do_full(c), last & 1, a.wait_limit_ns);
        }
      }
    }
  } else if (warp == 5 || warp == 6) {
    // Two MMA issuers: A (warp 5) issues S = Q K^T and dK^T += Q^T dS (the Q
    // operand), B (warp 6) issues dP = dO V^T and dV^T += dO^T P (the dO operand).
    // P needs only S, so dV^T(i) starts while the softmax side still computes
    // dS(i) = P (dP - D); dK^T(i) follows once dS(i) is written.  A issues
    // S(i+1) (the other Q stage) as soon as the softmax side has read S(i),
    // before dK^T(i), so the next tile's exponentials overlap this tile's products.
    if (lane == 0) {
      const bool is_a = warp == 5;
      constexpr uint32_t id_s = idesc_bf16(128, BN, false, false);  // S, dP: [128 q x BN]
      constexpr uint32_t id_t = idesc_bf16(128, BN, true, true);    // dV^T, dK^T: [128 h x BN]
      const uint64_t d_k = sdesc_sw128(sbase + C::k_off, 16, 1024);
      const uint64_t d_v = sdesc_sw128(sbase + C::v_off, 16, 1024);
      const uint64_t d_do = sdesc_sw128(sbase + C::do_off, 16, 1024);
      const uint64_t d_z = sdesc_sw128(sbase + (is_a ? C::ds_off : C::p_off), kQChunk, 1024);
      const uint32_t acc_col = is_a ? C::dk_col : C::dv_col;         // dK^T or dV^T
      bool ok = true;
      // S(n) = Q(n) K^T from Q stage n % QB.
      auto issue_s = [&](int n) -> bool {
        const int qb = n % QB;
        const uint64_t d_q = sdesc_sw128(sbase + C::q_off + qb * HC * kQChunk, 16, 1024);
        for (int c = 0; c < HC; ++c) {
          if (!mbar_wait(q_full(qb, c), (n / QB) & 1, ab)) return false;
          tc_fence_after();
          const uint64_t xa = sdesc_add(d_q, c * kQChunk), yb = sdesc_add(d_k, c * C::KV_CHUNK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + C::s_col, sdesc_add(xa, kk * 32), sdesc_add(yb, kk * 32), id_s,
                   (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(s_full);
        return true;
      };
      // dK^T (dV^T) += X^T Z over the 128 packed query rows: X = Q of tile n's
      // stage (or dO), Z = dS (or P); releases X half by half.
      auto issue_acc = [&](int n, uint32_t x_off) {
        const uint64_t d_xT = sdesc_sw128(sbase + x_off, kQChunk, 1024);  // X^T, MN-major
        for (int h = 0; h < HH; ++h) {
          const uint64_t xA = sdesc_add(d_xT, 2 * h * kQChunk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + acc_col + h * BN, sdesc_add(xA, kk * 2048), sdesc_add(d_z, kk * 2048), id_t,
                   (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(is_a ? q_empty(n % QB, h) : do_empty(h));
        }
      };
      // next non-empty Q tile after qt (qrng.y if none)
      auto next_tile = [&](int qt) {
        for (++qt; qt < qrng.y; ++qt)
          if (tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) != TILE_EMPTY) break;
        return qt;
      };
      int i = 0;
      for (int qt = qrng.x; qt < qrng.y && ok; ++qt) {
        if (tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN) == TILE_EMPTY) continue;
        if (i == 0 && !mbar_wait(kv_full, 0, ab)) { ok = false; break; }
        if (is_a) {
          if (i == 0 && !issue_s(0)) { ok = false; break; }
          const bool more = next_tile(qt) < qrng.y;
          // S(i+1) overwrites S(i) in TMEM: after the softmax side read it (p_full).
          if (more && (!mbar_wait(p_full, i & 1, ab) || !issue_s(i + 1))) { ok = false; break; }
          if (!mbar_wait(ds_full, i & 1, ab)) { ok = false; break; }
          tc_fence_after();
          issue_acc(i, C::q_off + (i % QB) * HC * kQChunk);
        } else {
          // dP(i-1) is read by the softmax side until it signals dS(i-1).
          if (i > 0 && !mbar_wait(ds_full, (i - 1) & 1, ab)) { ok = false; break; }
          for (int c = 0; c < HC && ok; ++c) {
            if (!mbar_wait(do_full(c), i & 1, ab)) { ok = false; break; }
            tc_fence_after();
            const uint64_t xa = sdesc_add(d_do, c * kQChunk);
            const uint64_t yb = sdesc_add(d_v, c * C::KV_CHUNK);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + C::dp_col, sdesc_add(xa, kk * 32), sdesc_add(yb, kk * 32), id_s,
                     (c > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(dp_full);
          if (!mbar_wait(p_full, i & 1, ab)) { ok = false; break; }
          tc_fence_after();
          issue_acc(i, C::do_off);
        }
        ++i;
      }
      if (!ok) {
        mma_commit(teardown(is_a ? 0 : 1));
        mbar_wait_teardown(teardown(is_a ? 0 : 1), 0, a.wait_limit_ns);
      }
    }
  } else {
    // Softmax side: the row reads TMEM lane quadrant warp % 4; the two warps of
    // a quadrant split the key columns (no row reduction is needed: lse and D
    // are precomputed).
    const int quad = warp & 3, half = warp >= 7 ? 1 : 0;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    constexpr int NCH = BN / 64;  // 32-column chunks per warp
    bool ok = true;
    int i = 0;
    for (int qt = qrng.x; qt < qrng.y; ++qt) {
      const int cls = tile_class(a, qr, kr, b, bk % a.K, qt, jt, Tb, BN);
      if (cls == TILE_EMPTY) continue;
      const int g = r / Tb, t = qt * Tb + (r - g * Tb);
      const bool valid = t < a.T;  // rows past T (ragged last tile) are inert
      const long row = ((long)bk * a.G + g) * a.T + t;
      const float lse = valid ? a.lse[row] : -INFINITY;
      const float lse2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
      const float Dr = valid ? a.delta[row] : 0.f;
      const int my_seg = (a.seg_q && valid) ? a.seg_q[(long)b * a.T + t] : 0;
      RowKeep keep{};
      if constexpr (SEGS)
        if (cls == TILE_PARTIAL) keep = row_keep(a, b, jt, s0, t, my_seg);
      // Phase 1: P = exp(S - lse) once S(i) is done, computed into registers
      // first; the P buffer is then overwritten once its reader dV^T(i-1)
      // (issuer B's) is done.
      if (!warp_wait(s_full, i & 1, ab)) { ok = false; break; }
      tc_fence_after();
      uint32_t pp[NCH][16];  // this warp's P (bf16 pairs), kept for phase 2
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = half * NCH + cc;
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + C::s_col + c * 32, sv);
        tmem_wait_ld();
        float* sf = reinterpret_cast<float*>(sv);
        if (cls == TILE_PARTIAL)
          mask32<SEGS>(*reinterpret_cast<float(*)[32]>(sf), a, b, bk % a.K, g, t, my_seg, s0 + c * 32, s0, keep);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pp[cc][k] = pack_bf16x2(fast_exp2(fmaf(sf[2 * k], kLog2e, -lse2)),
                                  fast_exp2(fmaf(sf[2 * k + 1], kLog2e, -lse2)));
      }
      if (i > 0 && !wait_halves<HH>(do_empty, (i - 1) & 1, ab)) { ok = false; break; }
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) store_row32(sm + C::p_off, r, half * NCH + cc, pp[cc]);
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor cores
      tc_fence_before();
      mbar_arrive(p_full);
      // Phase 2: dS = P (dP - D) once dP(i) is done (masked entries have P = 0).
      // The dS buffer's reader is dK^T(i-1), which A issued after S(i), so its
      // release barrier is waited for.
      if (!warp_wait(dp_full, i & 1, ab)) { ok = false; break; }
      if (i > 0) {
        const int pq = (i - 1) % QB;
        if (!wait_halves<HH>([&](int h) { return q_empty(pq, h); }, ((i - 1) / QB) & 1, ab)) { ok = false; break; }
      }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int c = half * NCH + cc;
        uint32_t pv[32], dd[16];
        tmem_ld32(tmem + lane_base + C::dp_col + c * 32, pv);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 pk = unpack_bf16x2(pp[cc][k]);
          dd[k] = pack_bf16x2(pk.x * (__uint_as_float(pv[2 * k]) - Dr),
                              pk.y * (__uint_as_float(pv[2 * k + 1]) - Dr));
        }
        store_row32(sm + C::ds_off, r, c, dd);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);
      ++i;
    }
    // Epilogue: lanes carry the head dim, columns the keys.
    const int lq = (i - 1) % QB;  // Q stage of the last tile
    const bool have = i > 0 && ok &&
                      wait_halves<HH>([&](int h) { return q_empty(lq, h); }, ((i - 1) / QB) & 1, ab) &&
                      wait_halves<HH>(do_empty, (i - 1) & 1, ab);
    if (have) tc_fence_after();
    dkdv_epilogue<H, BN, SPLIT>(a, tmem + lane_base + C::dv_col, tmem + lane_base + C::dk_col, r, half,
                                have, jt, split, bk, reinterpret_cast<volatile int*>(sm + C::misc_off + 16));
  }
  if (tid == 0) mbar_wait_teardown(kv_full, 0, a.wait_limit_ns);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// D[row] = sum_h dO[row, h] * o[row, h] in fp32.  H / 8 lanes share a row
// (one 16-byte load of o and of dO each); a warp covers 32 / (H / 8) rows per
// step and takes kPreSteps steps with all loads issued before any is used, so
// each warp keeps 2 * kPreSteps loads in flight.  HBM-bound.
constexpr int kPreSteps = 4;
template <int H>
__global__ void bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                      const __nv_bfloat16* __restrict__ dO, float* __restrict__ delta,
                                      long rows, int* __restrict__ zero, int n_zero) {
  constexpr int TPR = H / 8, RPW = 32 / TPR;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero[i] = 0;
  const int lane = threadIdx.x & 31;
  const long warp_id = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const long row0 = warp_id * kPreSteps * RPW + lane / TPR;
  const int col = lane % TPR;
  uint4 x[kPreSteps], d[kPreSteps];
#pragma unroll
  for (int u = 0; u < kPreSteps; ++u) {
    const long row = row0 + (long)u * RPW;
    if (row < rows) {
      x[u] = __ldg(reinterpret_cast<const uint4*>(o + row * H) + col);
      d[u] = __ldg(reinterpret_cast<const uint4*>(dO + row * H) + col);
    } else {
      x[u] = make_uint4(0, 0, 0, 0);
      d[u] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int u = 0; u < kPreSteps; ++u) {
    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&x[u]);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d[u]);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fx = __bfloat1622float2(x2[j]);
      const float2 fd = __bfloat1622float2(d2[j]);
      acc = fmaf(fx.x, fd.x, acc);
      acc = fmaf(fx.y, fd.y, acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const long row = row0 + (long)u * RPW;
    if (col == 0 && row < rows) delta[row] = acc;
  }
}

// Per-tile [min, max] of segment ids: one warp per (b, tile).  With `runs`
// (the KV tiles), also each tile's segment-run byte (see kRunsGeneral).
__global__ void seg_ranges_kernel(const int32_t* __restrict__ seg, int L, int tile, int n_tiles,
                                  long total, int2* __restrict__ out, uint8_t* __restrict__ runs) {
  const long w = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= total) return;
  const long b = w / n_tiles;
  const int j = (int)(w - b * n_tiles);
  const int32_t* p = seg + b * L + (long)j * tile;
  const int n = min(tile, L - j * tile);  // the last tile may be ragged
  int mn = INT_MAX, mx = INT_MIN;
  int changes = 0, pos = tile, prev_last = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {  // uniform over the warp
    const int i = i0 + lane;
    const int v = __ldg(p + min(i, n - 1));  // past the end: the last id again
    mn = min(mn, v);
    mx = max(mx, v);
    const int left = __shfl_up_sync(0xffffffffu, v, 1);
    const bool change = i > 0 && i < n && v != (lane == 0 ? prev_last : left);
    const uint32_t m = __ballot_sync(0xffffffffu, change);
    if (m != 0u && changes == 0) pos = i0 + __ffs((int)m) - 1;  // first key of the second run
    changes += __popc(m);
    prev_last = __shfl_sync(0xffffffffu, v, 31);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    out[w] = make_int2(mn, mx);
    if (runs != nullptr)
      runs[w] = changes == 0 ? (uint8_t)tile : changes == 1 ? (uint8_t)pos : kRunsGeneral;
  }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes, int* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (*configured == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *configured = dev;
  return e;
}

template <int H, int BN, bool SEGS>
cudaError_t launch_dq_h(const BwdArgs& a, cudaStream_t st, bool overlap_previous) {
  static int configured = -1;
  cudaError_t e = set_smem(fa_bwd_dq_kernel<H, BN, SEGS>, DqCfg<H, BN>::alloc, &configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_qtiles * a.B * a.K);
  cfg.blockDim = dim3(kDqThreads);
  cfg.dynamicSmemBytes = DqCfg<H, BN>::alloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fa_bwd_dq_kernel<H, BN, SEGS>, a);
}
template <int H, int BN>
cudaError_t launch_dq_h(const BwdArgs& a, cudaStream_t st, bool overlap_previous) {
  return a.seg_q != nullptr ? launch_dq_h<H, BN, true>(a, st, overlap_previous)
                            : launch_dq_h<H, BN, false>(a, st, overlap_previous);
}

template <int H, int BN, bool SPLIT, bool SEGS>
cudaError_t launch_dkdv_h(const BwdArgs& a, cudaStream_t st) {
  static int configured = -1;
  cudaError_t e = set_smem(fa_bwd_dkdv_kernel<H, BN, SPLIT, SEGS>, DkvCfg<H, BN>::alloc, &configured);
  if (e != cudaSuccess) return e;
  fa_bwd_dkdv_kernel<H, BN, SPLIT, SEGS><<<dim3(a.n_kvtiles * (SPLIT ? a.q_splits : 1) * a.B * a.K),
                                           kThreads, DkvCfg<H, BN>::alloc, st>>>(a);
  return cudaGetLastError();
}
template <int H, int BN, bool SPLIT>
cudaError_t launch_dkdv_h(const BwdArgs& a, cudaStream_t st) {
  return a.seg_q != nullptr ? launch_dkdv_h<H, BN, SPLIT, true>(a, st) : launch_dkdv_h<H, BN, SPLIT, false>(a, st);
}

template <int H, int BN, bool SPLIT, bool SEGS>
cudaError_t launch_dkdv1_h(const BwdArgs& a, cudaStream_t st) {
  static int configured = -1;
  cudaError_t e = set_smem(fa_bwd_dkdv1_kernel<H, BN, SPLIT, SEGS>, Dkv1Cfg<H, BN>::alloc, &configured);
  if (e != cudaSuccess) return e;
  fa_bwd_dkdv1_kernel<H, BN, SPLIT, SEGS><<<dim3(a.n_kvtiles * (SPLIT ? a.q_splits : 1) * a.B * a.K),
                                            kThreads, Dkv1Cfg<H, BN>::alloc, st>>>(a);
  return cudaGetLastError();
}
template <int H, int BN, bool SPLIT>
cudaError_t launch_dkdv1_h(const BwdArgs& a, cudaStream_t st) {
  return a.seg_q != nullptr ? launch_dkdv1_h<H, BN, SPLIT, true>(a, st) : launch_dkdv1_h<H, BN, SPLIT, false>(a, st);
}

}  // namespace

BwdWorkspace bwd_workspace(int B, int K, int G, int T, int S, int H, int sm_count) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t d = up((size_t)B * K * G * T * sizeof(float));
  const size_t tb = kRows / G, kvr = kMinBwdKvRows;
  const size_t nq = (T + tb - 1) / tb, nk = (S + kvr - 1) / kvr;
  const size_t r = up((size_t)B * (nq + nk) * sizeof(int2));
  const size_t ru = up((size_t)B * nk);  // one segment-run byte per KV tile
  BwdWorkspace w{d, d + r, 0, 0, d + r + ru, d + r + ru};
  // Every KV tile size the backward may pick for H: the largest split part.
  size_t cnt = 0, part = 0;
  const size_t Hk = H < 128 ? 128 : H;  // the kernels' head dim (H = 64 runs as 128)
  for (int rows = 64; rows <= (H <= 128 ? 128 : 64); rows *= 2) {
    const long ctas = (long)B * K * ((S + rows - 1) / rows);
    if (ctas <= 0 || ctas >= sm_count) continue;
    cnt = std::max(cnt, up((size_t)ctas * sizeof(int)));
    part = std::max(part, (size_t)kMaxQSplits * ctas * 2 * rows * Hk * sizeof(float));
  }
  if (part > 0) {
    w.counters = w.base;
    w.partials = w.base + cnt;
    w.total = w.partials + up(part);
  }
  return w;
}

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* delta, long rows, int H,
                                  int* zero, int n_zero, cudaStream_t st) {
  const int warps = 8;
  auto go = [&](auto kern, int tpr) {
    const long rows_per_block = (long)warps * kPreSteps * (32 / tpr);
    const long blocks = (rows + rows_per_block - 1) / rows_per_block;
    kern<<<(unsigned)blocks, warps * 32, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(o),
                                                  reinterpret_cast<const __nv_bfloat16*>(dO), delta,
                                                  rows, zero, zero ? n_zero : 0);
  };
  switch (H) {
    case 64: go(bwd_preprocess_kernel<64>, 8); break;
    case 128: go(bwd_preprocess_kernel<128>, 16); break;
    case 256: go(bwd_preprocess_kernel<256>, 32); break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

cudaError_t launch_seg_ranges(const BwdArgs& a, cudaStream_t st) {
  if (a.seg_q == nullptr) return cudaSuccess;
  int2* qr = a.seg_ranges;
  int2* kr = qr + (long)a.B * a.n_qtiles;
  const int Tb = kRows / a.G;
  const long nq = (long)a.B * a.n_qtiles, nk = (long)a.B * a.n_kvtiles;
  const int warps = 8;
  seg_ranges_kernel<<<(unsigned)((nq + warps - 1) / warps), warps * 32, 0, st>>>(a.seg_q, a.T, Tb,
                                                                                a.n_qtiles, nq, qr, nullptr);
  seg_ranges_kernel<<<(unsigned)((nk + warps - 1) / warps), warps * 32, 0, st>>>(
      a.seg_kv, a.S, a.kv_rows, a.n_kvtiles, nk, kr, a.seg_runs);
  return cudaGetLastError();
}

// H = 64 runs the H = 128 kernels: the TMA boxes of the upper 64 head dims lie
// wholly past the tensors' last dim and arrive zero-filled, which adds zero to
// S and dP and gives zero rows of dK^T, dV^T and zero dQ columns, none of
// which is stored.
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t st) {
  const bool split = a.q_splits > 1;
  const bool h128 = a.H == 128 || a.H == 64;
  if (h128 && a.kv_rows == 128)
    return split ? launch_dkdv_h<128, 128, true>(a, st) : launch_dkdv_h<128, 128, false>(a, st);
  if (h128 && a.kv_rows == 64)
    return split ? launch_dkdv_h<128, 64, true>(a, st) : launch_dkdv_h<128, 64, false>(a, st);
  if (a.H == 256 && a.kv_rows == 64)
    return split ? launch_dkdv1_h<256, 64, true>(a, st) : launch_dkdv1_h<256, 64, false>(a, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t st, bool overlap_previous) {
  const bool h128 = a.H == 128 || a.H == 64;
  if (h128 && a.kv_rows == 128) return launch_dq_h<128, 128>(a, st, overlap_previous);
  if (h128 && a.kv_rows == 64) return launch_dq_h<128, 64>(a, st, overlap_previous);
  if (a.H == 256 && a.kv_rows == 64) return launch_dq_h<256, 64>(a, st, overlap_previous);
  return cudaErrorNotSupported;
}

}  // namespace fa
