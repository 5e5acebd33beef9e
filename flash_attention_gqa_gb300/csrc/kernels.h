// Internal interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Tile geometry shared by every kernel.
constexpr int kRows = 128;     // packed query rows per Q tile (G heads x 128/G positions)
constexpr int kKvRows = 128;   // key/value rows per KV tile in the forward
// 64-dim chunks the forward moves per K or V copy: the whole tile up to
// H = 128; at H = 256 one chunk, so the first products of a K tile can start
// while its other chunks are still landing.
constexpr int fwd_copy_chunks(int H) { return H >= 256 ? 1 : H / 64; }
constexpr int kMaxKvTiles = 1024;  // S <= 131072

// Segment-id layout of a KV tile, one byte per tile: the index of the key
// where the id changes when the tile's ids form at most two runs (the tile's
// key count when they form one), else kRunsGeneral.  Where it is not
// kRunsGeneral, the keys a query row keeps are one contiguous range.
constexpr uint8_t kRunsGeneral = 0xff;

// Block-sparse mask metadata (device pointers; cls == nullptr: no mask).
struct BlockMask {
  const uint8_t* cls;     // [heads, nqb, nkb] EMPTY / FULL / PARTIAL
  const int32_t* idx;     // [heads, nqb, nkb] bitmask index of PARTIAL blocks
  const uint32_t* bits;   // [n_partial, 128, 4]
  int heads;              // 1 or K*G
  int nqb, nkb;           // ceil(T / 128), ceil(S / 128)
};

struct FwdArgs {
  CUtensorMap tm_q;   // q as 4-D {H, T, G, B*K}, box {64, 128/G, G, 1}, 128B swizzle
  CUtensorMap tm_k;   // k as 4-D {64, S, H/64, B*K}, box {64, 128, fwd_copy_chunks(H), 1}
  CUtensorMap tm_v;   // v, same as k
  CUtensorMap tm_o;   // o, same geometry as q (TMA store of the finished tile)
  void* o;            // bf16 [B*K, G, T, H]
  float* lse;         // [B*K, G, T]
  const int32_t* seg_q;   // [B, T] or null
  const int32_t* seg_kv;  // [B, S] or null
  int B, K, G, T, S, H;
  int causal;
  int n_qtiles;       // ceil(T / (128 / G))
  BlockMask bm;
  int n_splits;       // > 1: split-KV mode (grid.z splits the KV-tile schedule)
  float* part_o;      // split-KV: fp32 [n_splits, B*K*G*T, H] partial outputs
  float* part_lse;    // split-KV: [n_splits, B*K*G*T] partial lse (natural log)
  uint32_t* err;      // device error word
  uint64_t wait_limit_ns;
};

struct BwdArgs {
  CUtensorMap tm_q;    // q  as 4-D, box {64, 128/G, G, 1}
  CUtensorMap tm_do;   // dO as 4-D, same box
  CUtensorMap tm_k;    // k as 3-D, box {64, kv_rows, 1}
  CUtensorMap tm_v;    // v as 3-D, box {64, kv_rows, 1}
  CUtensorMap tm_dq;   // dq as 4-D, same box as q (TMA store)
  const float* lse;    // [B*K, G, T]
  const float* delta;  // [B*K, G, T]  D = rowsum(dO * o)
  // Per-tile [min, max] segment ids (read only with segment ids): B * n_qtiles
  // Q-tile pairs, then B * n_kvtiles KV-tile pairs.  8-byte aligned.
  int2* seg_ranges;
  // Segment-run byte of each KV tile (see kRunsGeneral): B * n_kvtiles bytes.
  uint8_t* seg_runs;
  void* dq;            // bf16 [B*K, G, T, H]
  void* dk;            // bf16 [B*K, S, H]
  void* dv;            // bf16 [B*K, S, H]
  const int32_t* seg_q;
  const int32_t* seg_kv;
  int B, K, G, T, S, H;
  int causal;
  int n_qtiles;        // T / (128 / G)
  int n_kvtiles;       // S / kv_rows
  int kv_rows;         // keys per KV tile of the backward kernels (64 or 128)
  int q_splits;        // CTAs sharing one KV tile's Q range in dK/dV (1: no split)
  float* dkv_part;     // q_splits > 1: fp32 partial dV, dK per dK/dV CTA [CTA][2][kv_rows][H]
  int* dkv_count;      // q_splits > 1: finished CTAs per (KV tile, b*K); zero between calls
  BlockMask bm;
  uint32_t* err;
  uint64_t wait_limit_ns;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st, int schedule);
// Also zeroes n_zero ints at zero (the dK/dV split counters; may be null).
cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* delta, long rows, int H,
                                  int* zero, int n_zero, cudaStream_t st);
cudaError_t launch_seg_ranges(const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t st);
// overlap_previous: launch with programmatic stream serialization so the grid
// may start while the immediately preceding dK/dV grid (which triggers its
// dependents at start) is still running; only valid right after launch_bwd_dkdv.
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t st, bool overlap_previous);
cudaError_t launch_fill_empty(void* o, float* lse, long rows, int H, cudaStream_t st);
cudaError_t launch_split_combine(const float* part_o, const float* part_lse, int n_splits, void* o,
                                 float* lse, long rows, int H, cudaStream_t st);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st);

// KV rows per tile of the backward kernels.  H = 256 always takes 64 (a
// 128-key K/V pair does not fit in shared memory next to the Q/dO tiles); H <=
// 128 takes 128 unless that leaves the dK/dV grid (one CTA per KV tile and
// b*K) smaller than the GPU, where 64-key tiles double its CTAs.
inline int bwd_kv_rows(int H, int B, int K, int S, int sm_count) {
  if (H == 256) return 64;
  const long ctas = (long)B * K * ((S + 127) / 128);
  return ctas < sm_count ? 64 : 128;
}
constexpr int kMinBwdKvRows = 64;  // the workspace's range table is sized for it

// Q-range split of the dK/dV grid.  With fewer dK/dV CTAs than SMs, the Q
// tiles of each KV tile are dealt to q_splits CTAs (1..kMaxQSplits); 1 when the
// grid already fills the GPU.  H <= 128: the largest count that keeps the grid
// to one wave (a second wave of light CTAs, with their extra partial tiles to
// write and add, measured slower than longer sweeps: T=1024 backward 53.4 us at
// 4 splits, 46.8 us at 2).  H = 256, where a tile costs twice as much: the
// count minimising waves / splits, ties going to the larger count when the
// sweeps are uneven (causal, segment ids or a block mask: the first KV tiles'
// sweeps are the longest) and to the smaller otherwise.
constexpr int kMaxQSplits = 4;
inline int bwd_q_splits(long ctas, int sm_count, bool uneven, int H) {
  if (ctas <= 0 || ctas >= sm_count) return 1;
  if (H <= 128) {
    int n = 1;
    while (n < kMaxQSplits && ctas * (n + 1) <= sm_count) ++n;
    return n;
  }
  int best = 1;
  double best_cost = 1e30;
  for (int n = 1; n <= kMaxQSplits; ++n) {
    const double cost = (double)((ctas * n + sm_count - 1) / sm_count) / n;
    if (cost < best_cost || (uneven && cost == best_cost)) { best_cost = cost; best = n; }
  }
  return best;
}

// Backward workspace: fp32 D rows, then per-tile segment-id ranges (the base
// part), then, where a Q-range split can apply (a dK/dV grid smaller than
// sm_count for some KV tile size), the split counters and kMaxQSplits fp32
// partial dK/dV tiles per dK/dV CTA.
struct BwdWorkspace {
  size_t ranges;    // offset of the segment-range table (256-byte aligned)
  size_t runs;      // offset of the KV tiles' segment-run bytes (256-byte aligned)
  size_t counters;  // offset of the split counters (0 where no split can apply)
  size_t partials;  // offset of the partial tiles
  size_t base;      // bytes without the split part
  size_t total;     // bytes with it
};
BwdWorkspace bwd_workspace(int B, int K, int G, int T, int S, int H, int sm_count);

}  // namespace fa
